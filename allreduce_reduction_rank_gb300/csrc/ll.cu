// ll.cu -- the all-pair LL-packet allreduce on one GPU.
//
// mscclpp commit history, the allreduce_allpair_packet fix: send, reduce and
// write-back run in the same thread block, the input buffer is never
// overwritten, and the reducer checks each packet's flag.  A packet is 8
// bytes: a 4-byte payload and a 4-byte epoch flag written together by one
// 8-byte store, so a reader that sees the flag also sees the payload.
//
//   pack          : rank r's input -> packets in pkts[r], flag = epoch
//   unpack_reduce : rank r polls packet group q of every rank k = 0..N-1 (in
//                   order) until the flags equal epoch, adds the payloads in
//                   binary32, rounds once and writes the elements to all N
//                   outputs.
//
// Threads move 16 bytes of payload (4 packets, 32 bytes of packet buffer) at
// a time with two 16-byte accesses; each 16-byte access is two
// single-copy-atomic 8-byte packets.  Every poll is bounded: after max_spins
// re-reads the thread records SAR_ERR_TIMEOUT in the caller's status word and
// returns, and every other thread that has to wait returns as soon as it sees
// a non-zero status.
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

constexpr unsigned kMaxSleepNs = 1024;

__device__ __forceinline__ int32_t ld_status(const int32_t* s) {
    int32_t v;
    asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(s) : "memory");
    return v;
}

// Wait until four consecutive packets (already loaded into w) carry `epoch`.
// Returns false when this thread gave up or saw another thread give up.
__device__ __forceinline__ bool poll_quad(const uint64_t* src, uint32_t epoch, uint64_t max_spins, int32_t* status,
                          uint64_t (&w)[4]) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        if (packet_flag(w[0]) == epoch && packet_flag(w[1]) == epoch && packet_flag(w[2]) == epoch &&
            packet_flag(w[3]) == epoch)
            return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        if (ld_status(status) != 0) return false;
        __nanosleep(ns);
        if (ns < kMaxSleepNs) ns *= 2;
        ld_packets2(src, w[0], w[1]);
        ld_packets2(src + 2, w[2], w[3]);
    }
}

__device__ __forceinline__ bool poll_one(const uint64_t* src, uint32_t epoch, uint64_t max_spins, int32_t* status,
                         uint64_t& w) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        if (packet_flag(w) == epoch) return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        if (ld_status(status) != 0) return false;
        __nanosleep(ns);
        if (ns < kMaxSleepNs) ns *= 2;
        w = ld_packet(src);
    }
}

// ---------------------------------------------------------------------------
// Pack.  p.in[r] = input, p.out[r] = packet buffer of rank r.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
ll_pack_vec_kernel(const RankPtrs p, size_t nbytes, uint32_t epoch) {
    pdl_wait();
    const int r = blockIdx.y;
    const uint4* src = static_cast<const uint4*>(p.in[r]);
    uint64_t* dst = static_cast<uint64_t*>(p.out[r]);
    const size_t nq = nbytes / 16;
    for (size_t q = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; q < nq;
         q += static_cast<size_t>(gridDim.x) * kThreads) {
        const uint4 x = ld_stream(src + q);
        st_packets2(dst + 4 * q, make_packet(x.x, epoch), make_packet(x.y, epoch));
        st_packets2(dst + 4 * q + 2, make_packet(x.z, epoch), make_packet(x.w, epoch));
    }
    // Up to 4 packets after the last whole 16 bytes; the last may be padded.
    if (blockIdx.x == 0 && threadIdx.x < 4) {
        const size_t w = 4 * nq + threadIdx.x;
        if (4 * w < nbytes) {
            const unsigned char* b = static_cast<const unsigned char*>(p.in[r]);
            uint32_t payload = 0;
            for (int k = 0; k < 4; ++k)
                if (4 * w + k < nbytes) payload |= static_cast<uint32_t>(b[4 * w + k]) << (8 * k);
            st_packet(dst + w, make_packet(payload, epoch));
        }
    }
}

// Inputs that are not 16-byte aligned: one packet per thread, byte loads.
__global__ void __launch_bounds__(kThreads)
ll_pack_bytes_kernel(const RankPtrs p, size_t nbytes, uint32_t epoch) {
    pdl_wait();
    const int r = blockIdx.y;
    const unsigned char* b = static_cast<const unsigned char*>(p.in[r]);
    uint64_t* dst = static_cast<uint64_t*>(p.out[r]);
    const size_t npk = (nbytes + 3) / 4;
    for (size_t w = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; w < npk;
         w += static_cast<size_t>(gridDim.x) * kThreads) {
        uint32_t payload = 0;
        for (int k = 0; k < 4; ++k)
            if (4 * w + k < nbytes) payload |= static_cast<uint32_t>(b[4 * w + k]) << (8 * k);
        st_packet(dst + w, make_packet(payload, epoch));
    }
}

// ---------------------------------------------------------------------------
// Poll + unpack + reduce + write-back.  p.in[k] = packet buffer of rank k,
// p.out[j] = output of rank j.  Rank r (blockIdx.y) owns packet groups
// [r*chunk_q, min(nq, (r+1)*chunk_q)), a group being 4 packets = 16 payload
// bytes.
// ---------------------------------------------------------------------------
template <int DT, int NR>
__global__ void __launch_bounds__(kThreads)
ll_unpack_reduce_kernel(const RankPtrs p, int n_rt, size_t count, size_t nbytes, size_t chunk_q, uint32_t epoch,
                        uint64_t max_spins, int32_t* status, bool vec_out) {
    pdl_wait();
    constexpr int VE = Elem<DT>::kVE;
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR == 0 ? 4 : (NR < 8 ? NR : 8);
    const int n = ranks<NR>(n_rt);
    const int r = blockIdx.y;
    const size_t npk = (nbytes + 3) / 4;
    const size_t nq = (npk + 3) / 4;
    const size_t qb = static_cast<size_t>(r) * chunk_q;
    if (qb >= nq) return;
    const size_t qe = min(nq, qb + chunk_q);

    for (size_t q = qb + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; q < qe;
         q += static_cast<size_t>(gridDim.x) * kThreads) {
        if (16 * (q + 1) <= nbytes) {
            // A whole group: 4 packets of payload from every rank.
            Acc<DT> acc;
// Windows of 8 ranks run as a loop (one window for up to 8 ranks).
#pragma unroll 1
            for (int k0 = 0; k0 < n; k0 += WIN) {
                uint64_t w[WIN][4];
#pragma unroll
                for (int k = 0; k < WIN; ++k) {
                    if (NR == 0 && k0 + k >= n) break;
                    const uint64_t* src = static_cast<const uint64_t*>(p.in[k0 + k]) + 4 * q;
                    ld_packets2(src, w[k][0], w[k][1]);
                    ld_packets2(src + 2, w[k][2], w[k][3]);
                }
#pragma unroll
                for (int k = 0; k < WIN; ++k) {
                    if (NR == 0 && k0 + k >= n) break;
                    const uint64_t* src = static_cast<const uint64_t*>(p.in[k0 + k]) + 4 * q;
                    if (!poll_quad(src, epoch, max_spins, status, w[k])) return;
                    const uint4 x = make_uint4(packet_payload(w[k][0]), packet_payload(w[k][1]),
                                               packet_payload(w[k][2]), packet_payload(w[k][3]));
                    if (k0 + k == 0) acc_seed<DT>(acc, x);
                    else acc_add<DT>(acc, x);
                }
            }
            if (vec_out) {
                const uint4 y = acc_round<DT>(acc);
#pragma unroll
                for (int j = 0; j < n; ++j) st_stream(static_cast<uint4*>(p.out[j]) + q, y);
            } else {
#pragma unroll
                for (int e = 0; e < VE; ++e)
#pragma unroll
                    for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], q * VE + e, acc.v[e]);
            }
        } else {
            // The last group: 1..4 packets, the last one possibly padded.
            const size_t wend = min(npk, 4 * q + 4);
            for (size_t w = 4 * q; w < wend; ++w) {
                float acc[EP];
                for (int k = 0; k < n; ++k) {
                    const uint64_t* src = static_cast<const uint64_t*>(p.in[k]) + w;
                    uint64_t pk = ld_packet(src);
                    if (!poll_one(src, epoch, max_spins, status, pk)) return;
                    float x[EP];
                    widen_word<DT>(packet_payload(pk), x);
#pragma unroll
                    for (int e = 0; e < EP; ++e) acc[e] = (k == 0) ? x[e] : __fadd_rn(acc[e], x[e]);
                }
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    const size_t i = w * EP + e;
                    if (i < count)
                        for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], i, acc[e]);
                }
            }
        }
    }
}

inline unsigned grid_x(size_t items, size_t cap) {
    size_t g = (items + kThreads - 1) / kThreads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

constexpr size_t kGridCap = 65535;

template <int DT, int NR>
cudaError_t unpack_dispatch(int nranks, const RankPtrs& p, size_t count, uint32_t epoch, uint64_t max_spins,
                            int32_t* status, bool vec_out, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4, nq = (npk + 3) / 4;
    const size_t chunk_q = (nq + nranks - 1) / nranks;
    const dim3 grid(grid_x(chunk_q, kGridCap), nranks);
    launch_kernel(ll_unpack_reduce_kernel<DT, NR>, grid, dim3(kThreads), s, p, nranks, count, nbytes, chunk_q,
                  epoch, max_spins, status, vec_out);
    return cudaGetLastError();
}

template <int DT>
cudaError_t unpack_ranks(int nranks, const RankPtrs& p, size_t count, uint32_t epoch, uint64_t max_spins,
                         int32_t* status, bool vec_out, cudaStream_t s) {
    switch (nranks) {
    case 1: return unpack_dispatch<DT, 1>(1, p, count, epoch, max_spins, status, vec_out, s);
    case 2: return unpack_dispatch<DT, 2>(2, p, count, epoch, max_spins, status, vec_out, s);
    case 4: return unpack_dispatch<DT, 4>(4, p, count, epoch, max_spins, status, vec_out, s);
    case 8: return unpack_dispatch<DT, 8>(8, p, count, epoch, max_spins, status, vec_out, s);
    case 16: return unpack_dispatch<DT, 16>(16, p, count, epoch, max_spins, status, vec_out, s);
    case 32: return unpack_dispatch<DT, 32>(32, p, count, epoch, max_spins, status, vec_out, s);
    default:
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        return unpack_dispatch<DT, 0>(nranks, p, count, epoch, max_spins, status, vec_out, s);
    }
}

}  // namespace

cudaError_t launch_ll_pack(int nranks, const RankPtrs& p, size_t bytes, uint32_t epoch, bool vec,
                           cudaStream_t stream) {
    if (vec) {
        const dim3 grid(grid_x(bytes / 16 + 1, kGridCap), nranks);
        launch_kernel(ll_pack_vec_kernel, grid, dim3(kThreads), stream, p, bytes, epoch);
    } else {
        const dim3 grid(grid_x((bytes + 3) / 4, kGridCap), nranks);
        launch_kernel(ll_pack_bytes_kernel, grid, dim3(kThreads), stream, p, bytes, epoch);
    }
    return cudaGetLastError();
}

cudaError_t launch_ll_unpack_reduce(sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                                    uint32_t epoch, uint64_t max_spins, int32_t* status, bool vec_out,
                                    cudaStream_t stream) {
#define SAR_UNPACK(T) unpack_ranks<T>(nranks, p, count, epoch, max_spins, status, vec_out, stream)
    switch (dt) {
    case SAR_BF16: return SAR_UNPACK(SAR_BF16);
    case SAR_FP16: return SAR_UNPACK(SAR_FP16);
    case SAR_FP32: return SAR_UNPACK(SAR_FP32);
    case SAR_FP8_E4M3FN: return SAR_UNPACK(SAR_FP8_E4M3FN);
    case SAR_FP8_E4M3B15: return SAR_UNPACK(SAR_FP8_E4M3B15);
    }
#undef SAR_UNPACK
    return cudaErrorInvalidValue;
}

}  // namespace sar
