// ll_cta.cu -- the LL all-pair allreduce of a small call inside one CTA:
// the packets of every simulated rank live in that CTA's shared memory.
//
// mscclpp commit history, the allreduce_allpair_packet fix: send, reduce and
// write-back in the same thread block, packets checked by their flags.  When
// all N ranks' packets of a call fit one CTA's shared memory, that CTA plays
// every rank:
//
//   clear  : the CTA clears the packet slots [rank k][packet w] and
//            synchronises once;
//   send   : rank k's input words become packets {payload, flag} in slots
//            [k][*] (one 16-byte input vector -> 4 packets per item, items
//            spread over all threads);
//   reduce : thread t polls packet w = t, t + T, ... of every rank until its
//            flag is set (bounded; a timeout goes to the status word, if
//            any), adds the payloads in rank order 0..N-1 in binary32, rounds
//            once and writes the result to all N outputs.
//
// No packet leaves the SM, nothing is kept between calls (the slots start
// every launch at zero, so the flag is always 1), and the call is one launch.
// The reduce assigns packets to threads without regard to which rank's chunk
// they belong to: every element is reduced on its own, so the values are
// those of the chunked forms.
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

}  // namespace sar
