// ll_cta.cu -- the LL all-pair allreduce with the packets of every simulated
// rank in the shared memory of the CTA that makes and polls them.
//
// mscclpp commit history, the allreduce_allpair_packet fix: send, reduce and
// write-back in the same thread block, packets checked by their flags.  Here
// a CTA plays every rank for its share of the data:
//
//   clear  : the CTA clears its packet slots [rank k][packet w] and
//            synchronises once;
//   send   : rank k's input words become packets {payload, flag} in slots
//            [k][*] (one 16-byte input vector -> 4 packets per item, items
//            spread over the threads);
//   reduce : each thread polls its packets of every rank until their flags
//            are set (bounded; a timeout goes to the status word, if any),
//            adds the payloads in rank order 0..N-1 in binary32, rounds once
//            and writes the result to all N outputs.
//
// Two grids: cta_kernel, one CTA for a whole small call, and slice_kernel,
// one CTA per slice of the packets (the same packet range of every rank), so
// that a call of any size spreads over the SMs.  No packet leaves the SM,
// nothing is kept between calls (the slots start every launch at zero, so the
// flag is always 1), and a call is one launch.  The reduce assigns packets to
// threads without regard to which rank's chunk they belong to: every element
// is reduced on its own, so the values are those of the chunked forms.
#include "ll_packets.cuh"
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace llt {

constexpr int kCtaThreads = 512;
constexpr uint32_t kFlag = 1;
constexpr uint64_t kSpinPolls = 16;
constexpr unsigned kMaxSleepNs = 1024;

__device__ __forceinline__ void st_slot4(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.cta.shared.v2.u64 [%0], {%1, %2};"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_slot(uint64_t* p, uint64_t a) {
    asm volatile("st.relaxed.cta.shared.u64 [%0], %1;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "l"(a) : "memory");
}
__device__ __forceinline__ uint64_t ld_slot(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.cta.shared.u64 %0, [%1];"
                 : "=l"(v) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))) : "memory");
    return v;
}
__device__ __forceinline__ void ld_slot2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.cta.shared.v2.u64 {%0, %1}, [%2];"
                 : "=l"(a), "=l"(b) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))) : "memory");
}
__device__ __forceinline__ uint64_t packet(uint32_t payload) {
    return static_cast<uint64_t>(payload) | (static_cast<uint64_t>(kFlag) << 32);
}

template <int DT, int NR>
__global__ void __launch_bounds__(kCtaThreads)
cta_kernel(const RankPtrs p, int n_rt, size_t count, size_t nbytes, uint64_t max_spins, int32_t* status, bool in16,
           bool out16) {
    extern __shared__ __align__(16) uint64_t slots[];   // [rank k][npk]
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR > 0 ? (NR < 8 ? NR : 8) : 8;
    const int n = ranks<NR>(n_rt);
    const size_t npk = (nbytes + 3) / 4;
    const size_t stride = (npk + 1) / 2 * 2;            // slots per rank, even: 16-byte aligned rows
    for (size_t i = threadIdx.x; i < static_cast<size_t>(n) * stride; i += kCtaThreads) slots[i] = 0;
    __syncthreads();
    pdl_wait();

    // send: item = (rank k, group g of 4 packets).  (Loading several items
    // before storing their packets measured slower here.)
    const size_t ng = (npk + 3) / 4;
    for (size_t it = threadIdx.x; it < static_cast<size_t>(n) * ng; it += kCtaThreads) {
        const int k = static_cast<int>(it / ng);
        const size_t g = it % ng, w = 4 * g;
        const unsigned char* src = static_cast<const unsigned char*>(p.in[k]);
        uint64_t* row = slots + static_cast<size_t>(k) * stride;
        if (in16 && 16 * (g + 1) <= nbytes) {
            const uint4 q = ld_stream(reinterpret_cast<const uint4*>(src) + g);
            st_slot4(row + w, packet(q.x), packet(q.y));
            st_slot4(row + w + 2, packet(q.z), packet(q.w));
        } else {
            for (int m = 0; m < 4 && w + m < npk; ++m) st_slot(row + w + m, packet(payload_word(src, nbytes, w + m)));
        }
    }

    // reduce: packets w = t, t + T, ...; ranks in windows of up to 8, each
    // window's packets polled together.
    for (size_t w = threadIdx.x; w < npk; w += kCtaThreads) {
        float acc[EP];
        bool ok = true;
#pragma unroll 1
        for (int k0 = 0; k0 < n && ok; k0 += WIN) {
            uint64_t pk[WIN];
#pragma unroll
            for (int k = 0; k < WIN; ++k)
                if (k0 + k < n) pk[k] = ld_slot(slots + static_cast<size_t>(k0 + k) * stride + w);
            unsigned ns = 32;
            for (uint64_t spin = 0;; ++spin) {
                bool ready = true;
#pragma unroll
                for (int k = 0; k < WIN; ++k)
                    if (k0 + k < n) ready = ready && static_cast<uint32_t>(pk[k] >> 32) == kFlag;
                if (ready) break;
                if (spin >= max_spins) {
                    if (status != nullptr) atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
                    ok = false;
                    break;
                }
                if (spin >= kSpinPolls) {
                    __nanosleep(ns);
                    if (ns < kMaxSleepNs) ns *= 2;
                }
#pragma unroll
                for (int k = 0; k < WIN; ++k)
                    if (k0 + k < n && static_cast<uint32_t>(pk[k] >> 32) != kFlag)
                        pk[k] = ld_slot(slots + static_cast<size_t>(k0 + k) * stride + w);
            }
            if (!ok) break;
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (k0 + k >= n) break;
                float x[EP];
                widen_word<DT>(static_cast<uint32_t>(pk[k]), x);
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[e] = (k0 + k == 0) ? x[e] : __fadd_rn(acc[e], x[e]);
            }
        }
        if (!ok) break;
        if (out16 && 4 * (w + 1) <= nbytes) {
            const uint32_t y = narrow_word<DT>(acc);
            for (int j = 0; j < n; ++j) st_stream_word(static_cast<uint32_t*>(p.out[j]) + w, y);
        } else {
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const size_t i = w * EP + e;
                if (i < count)
                    for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], i, acc[e]);
            }
        }
    }
}

template <int DT, int NR>
cudaError_t cta_dispatch(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status,
                         bool in16, bool out16, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    const size_t smem = static_cast<size_t>(nranks) * ((npk + 1) / 2 * 2) * 8;
    if (smem > kLLCtaMaxSlotBytes) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(cta_kernel<DT, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kLLCtaMaxSlotBytes));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kCtaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cta_kernel<DT, NR>, p, nranks, count, nbytes, max_spins, status, in16, out16);
}

template <int DT>
cudaError_t cta_ranks(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status, bool in16,
                      bool out16, cudaStream_t s) {
    switch (nranks) {
    case 2: return cta_dispatch<DT, 2>(2, p, count, max_spins, status, in16, out16, s);
    case 4: return cta_dispatch<DT, 4>(4, p, count, max_spins, status, in16, out16, s);
    case 8: return cta_dispatch<DT, 8>(8, p, count, max_spins, status, in16, out16, s);
    default:
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        return cta_dispatch<DT, 0>(nranks, p, count, max_spins, status, in16, out16, s);
    }
}


// ---------------------------------------------------------------------------
// Sliced form: CTA b plays every rank for packets [b*SP, (b+1)*SP) of the
// buffers (SP = PPT*CT packets per rank), so a call of any size spreads over
// the SMs and no packet leaves the SM that made it.
//
//   clear  : the CTA clears its slots [rank k][SP] and synchronises once;
//   send   : item (k, g) turns input vector g of the slice of rank k into 4
//            packets in slots [k][4g..4g+3]; the items are spread over the
//            threads (rotated by a warp per rank), each thread issuing the
//            loads of up to 8 items before their packet stores;
//   reduce : thread t polls packets PPT*t .. PPT*t+PPT-1 of every rank (ranks
//            in windows of up to 8, each window's packets polled together)
//            until their flags are set, adds the payloads in rank order
//            0..N-1 in binary32, rounds once and writes the result (16 bytes
//            for PPT = 4, 4 for PPT = 1) to all N outputs.
// ---------------------------------------------------------------------------
// Slot of packet q (0..SP-1) of a slice in its rank's row: packets 0-1 of
// every group of 4 in the first half of the row, packets 2-3 in the second,
// so that the 16-byte accesses of a warp (two packets of consecutive groups)
// are contiguous and free of bank conflicts.
template <int SP> __device__ __forceinline__ int slice_slot(int q) {
    return ((q & 3) >> 1) * (SP / 2) + (q >> 2) * 2 + (q & 1);
}

template <int DT, int NR, int CT, int PPT>
__global__ void __launch_bounds__(CT)
slice_kernel(const RankPtrs p, int n_rt, size_t count, size_t nbytes, uint64_t max_spins, int32_t* status, bool in16,
             bool out16) {
    extern __shared__ __align__(16) uint64_t slots[];   // [rank k][slice_slot(q)]
    constexpr int SP = PPT * CT;
    constexpr int G = SP / 4;                           // input vectors per rank in a slice
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR > 0 ? (NR < 8 ? NR : 8) : 8;
    const int n = ranks<NR>(n_rt);
    const size_t npk = (nbytes + 3) / 4;
    const size_t w0 = static_cast<size_t>(blockIdx.x) * SP;
    const int np = static_cast<int>(min(static_cast<size_t>(SP), npk - w0));
    for (int i = threadIdx.x; i < n * SP; i += CT) slots[i] = 0;
    __syncthreads();
    pdl_wait();

    const int items = n * G;
    for (int u0 = 0; u0 * CT < items; u0 += 8) {
        uint32_t x[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int it = threadIdx.x + (u0 + u) * CT;
            const int k = it / G, g = (it + 32 * k) % G;
            if (it >= items || 4 * g >= np) continue;
            const size_t w = w0 + 4 * static_cast<size_t>(g);
            const unsigned char* src = static_cast<const unsigned char*>(p.in[k]);
            if (in16 && 4 * (w + 4) <= nbytes) {
                const uint4 q = ld_stream(reinterpret_cast<const uint4*>(src) + w / 4);
                x[u][0] = q.x; x[u][1] = q.y; x[u][2] = q.z; x[u][3] = q.w;
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) x[u][m] = 4 * g + m < np ? payload_word(src, nbytes, w + m) : 0;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int it = threadIdx.x + (u0 + u) * CT;
            const int k = it / G, g = (it + 32 * k) % G;
            if (it >= items || 4 * g >= np) continue;
            uint64_t* row = slots + k * SP;
            if (4 * g + 4 <= np) {
                st_slot4(row + slice_slot<SP>(4 * g), packet(x[u][0]), packet(x[u][1]));
                st_slot4(row + slice_slot<SP>(4 * g + 2), packet(x[u][2]), packet(x[u][3]));
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (4 * g + m < np) st_slot(row + slice_slot<SP>(4 * g + m), packet(x[u][m]));
            }
        }
    }

    const int t0 = PPT * threadIdx.x;   // first packet of this thread in the slice
    const int mn = np - t0;             // packets of this thread: min(PPT, mn)
    if (mn <= 0) return;
    float acc[PPT][EP];
    bool ok = true;
#pragma unroll 1
    for (int k0 = 0; k0 < n && ok; k0 += WIN) {
        uint64_t pk[WIN][PPT];
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
            const uint64_t* row = slots + (k0 + k) * SP;
            if (PPT == 4 && mn >= 4) {
                ld_slot2(row + slice_slot<SP>(t0), pk[k][0], pk[k][PPT > 1 ? 1 : 0]);
                ld_slot2(row + slice_slot<SP>(t0 + 2), pk[k][PPT > 2 ? 2 : 0], pk[k][PPT > 3 ? 3 : 0]);
            } else {
#pragma unroll
                for (int m = 0; m < PPT; ++m) pk[k][m] = m < mn ? ld_slot(row + slice_slot<SP>(t0 + m)) : packet(0);
            }
        }
        unsigned ns = 32;
        for (uint64_t spin = 0;; ++spin) {
            bool ready = true;
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (NR == 0 && k0 + k >= n) break;
#pragma unroll
                for (int m = 0; m < PPT; ++m) ready = ready && static_cast<uint32_t>(pk[k][m] >> 32) == kFlag;
            }
            if (ready) break;
            if (spin >= max_spins) {
                if (status != nullptr) atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
                ok = false;
                break;
            }
            if (spin >= kSpinPolls) {
                __nanosleep(ns);
                if (ns < kMaxSleepNs) ns *= 2;
            }
#pragma unroll
            for (int k = 0; k < WIN; ++k) {
                if (NR == 0 && k0 + k >= n) break;
#pragma unroll
                for (int m = 0; m < PPT; ++m)
                    if (static_cast<uint32_t>(pk[k][m] >> 32) != kFlag)
                        pk[k][m] = ld_slot(slots + (k0 + k) * SP + slice_slot<SP>(t0 + m));
            }
        }
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
#pragma unroll
            for (int m = 0; m < PPT; ++m) {
                float x[EP];
                widen_word<DT>(static_cast<uint32_t>(pk[k][m]), x);
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[m][e] = (k0 + k == 0) ? x[e] : __fadd_rn(acc[m][e], x[e]);
            }
        }
    }
    if (!ok) return;
    const size_t w = w0 + t0;
    if (out16 && mn >= PPT && 4 * (w + PPT) <= nbytes) {
        if constexpr (PPT == 4) {
            const uint4 y = make_uint4(narrow_word<DT>(acc[0]), narrow_word<DT>(acc[1]), narrow_word<DT>(acc[2]),
                                       narrow_word<DT>(acc[3]));
            for (int j = 0; j < n; ++j) st_stream(static_cast<uint4*>(p.out[j]) + w / 4, y);
        } else {
#pragma unroll
            for (int m = 0; m < PPT; ++m) {
                const uint32_t y = narrow_word<DT>(acc[m]);
                for (int j = 0; j < n; ++j) st_stream_word(static_cast<uint32_t*>(p.out[j]) + w + m, y);
            }
        }
    } else {
        for (int m = 0; m < PPT && m < mn; ++m) {
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const size_t i = (w + m) * EP + e;
                if (i < count)
                    for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], i, acc[m][e]);
            }
        }
    }
}

template <int DT, int NR, int CT, int PPT>
cudaError_t slice_launch(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status, bool in16,
                         bool out16, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    const size_t slices = (npk + PPT * CT - 1) / (PPT * CT);
    if (slices > 0x7FFFFFFFull) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(nranks) * PPT * CT * 8;
    if (smem > kLLCtaMaxSlotBytes) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(slice_kernel<DT, NR, CT, PPT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kLLCtaMaxSlotBytes));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(slices));
    cfg.blockDim = dim3(CT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, slice_kernel<DT, NR, CT, PPT>, p, nranks, count, nbytes, max_spins, status, in16,
                              out16);
}

// Slices of 4 packets per thread (16-byte result stores) while they still
// give kSliceWideCtas CTAs and at most 8 ranks; else 1 packet per thread.
// CTAs of 128 threads: the slots take nranks x 4 KiB or nranks x 1 KiB.
#ifndef SLICE_WIDE_CTAS
#define SLICE_WIDE_CTAS 152
#endif
constexpr size_t kSliceWideCtas = SLICE_WIDE_CTAS;

template <int DT, int NR>
cudaError_t slice_dispatch(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status,
                           bool in16, bool out16, cudaStream_t s) {
    const size_t npk = (count * Elem<DT>::kSize + 3) / 4;
    if constexpr (NR <= 8) {
        if (nranks <= 8 && (npk + 511) / 512 >= kSliceWideCtas)
            return slice_launch<DT, NR, 128, 4>(nranks, p, count, max_spins, status, in16, out16, s);
    }
    return slice_launch<DT, NR, 128, 1>(nranks, p, count, max_spins, status, in16, out16, s);
}

template <int DT>
cudaError_t slice_ranks(int nranks, const RankPtrs& p, size_t count, uint64_t max_spins, int32_t* status, bool in16,
                        bool out16, cudaStream_t s) {
    switch (nranks) {
    case 1: return slice_dispatch<DT, 1>(1, p, count, max_spins, status, in16, out16, s);
    case 2: return slice_dispatch<DT, 2>(2, p, count, max_spins, status, in16, out16, s);
    case 4: return slice_dispatch<DT, 4>(4, p, count, max_spins, status, in16, out16, s);
    case 8: return slice_dispatch<DT, 8>(8, p, count, max_spins, status, in16, out16, s);
    case 16: return slice_dispatch<DT, 16>(16, p, count, max_spins, status, in16, out16, s);
    case 32: return slice_dispatch<DT, 32>(32, p, count, max_spins, status, in16, out16, s);
    default:
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        return slice_dispatch<DT, 0>(nranks, p, count, max_spins, status, in16, out16, s);
    }
}

}  // namespace llt

size_t ll_cta_slot_bytes(int nranks, size_t count, sar_dtype dt) {
    const size_t npk = (count * esize_of(dt) + 3) / 4;
    return static_cast<size_t>(nranks) * ((npk + 1) / 2 * 2) * 8;
}

cudaError_t launch_ll_cta(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                          int32_t* status, bool in16, bool out16, cudaStream_t stream) {
    switch (dt) {
    case SAR_BF16: return llt::cta_ranks<SAR_BF16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP16: return llt::cta_ranks<SAR_FP16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP32: return llt::cta_ranks<SAR_FP32>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3FN:
        return llt::cta_ranks<SAR_FP8_E4M3FN>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3B15:
        return llt::cta_ranks<SAR_FP8_E4M3B15>(nranks, p, count, max_spins, status, in16, out16, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_ll_slice(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                            int32_t* status, bool in16, bool out16, cudaStream_t stream) {
    switch (dt) {
    case SAR_BF16: return llt::slice_ranks<SAR_BF16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP16: return llt::slice_ranks<SAR_FP16>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP32: return llt::slice_ranks<SAR_FP32>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3FN:
        return llt::slice_ranks<SAR_FP8_E4M3FN>(nranks, p, count, max_spins, status, in16, out16, stream);
    case SAR_FP8_E4M3B15:
        return llt::slice_ranks<SAR_FP8_E4M3B15>(nranks, p, count, max_spins, status, in16, out16, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sar
