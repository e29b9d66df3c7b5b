// ll.cu -- the all-pair LL-packet allreduce on one GPU.
//
// mscclpp commit history, the allreduce_allpair_packet fix: send, reduce and
// write-back run in the same thread block, the input buffer is never
// overwritten, and the reducer checks each packet's flag.  A packet is 8
// bytes: a 4-byte payload and a 4-byte epoch flag written together by one
// 8-byte store, so a reader that sees the flag also sees the payload.
//
//   pack          : rank r's input -> packets in pkts[r], flag = epoch
//   unpack_reduce : rank r polls packet w of every rank k = 0..N-1 (in
//                   order) until the flags equal epoch, adds the payloads in
//                   binary32, rounds once and writes the elements to all N
//                   outputs.
//
// A pack thread turns 16 bytes of input into 4 packets (32 bytes of packet
// buffer): one 32-byte store when every packet buffer is 32-byte aligned, two
// 16-byte stores otherwise.  An unpack thread takes one packet index: an
// 8-byte load from each rank, all issued before the in-order adds.  A vector
// access is a set of single-copy-atomic 8-byte element accesses, so a packet's
// payload and flag are always written and read together.  Every poll is
// bounded: after max_spins re-reads the thread records SAR_ERR_TIMEOUT in the
// caller's status word and returns, and every other thread that has to wait
// returns as soon as it sees a non-zero status.
#include "ll_packets.cuh"
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

constexpr unsigned kMaxSleepNs = 1024;

// Wait until the packet (already loaded into w) carries `epoch`.  Returns
// false when this thread gave up or saw another thread give up.
__device__ __forceinline__ bool poll_one(const uint64_t* src, uint32_t epoch, uint64_t max_spins, int32_t* status,
                         uint64_t& w) {
    unsigned ns = 32;
    for (uint64_t spin = 0;; ++spin) {
        if (packet_flag(w) == epoch) return true;
        if (spin >= max_spins) {
            atomicCAS(status, 0, static_cast<int32_t>(SAR_ERR_TIMEOUT));
            return false;
        }
        if (ld_status_word(status) != 0) return false;
        __nanosleep(ns);
        if (ns < kMaxSleepNs) ns *= 2;
        w = ld_packet(src);
    }
}

// ---------------------------------------------------------------------------
// Pack.  p.in[r] = input, p.out[r] = packet buffer of rank r.  One 16-byte
// input vector per thread; kWide: every packet buffer is 32-byte aligned.
// ---------------------------------------------------------------------------
template <bool kWide>
__global__ void __launch_bounds__(kThreads)
ll_pack_vec_kernel(const RankPtrs p, size_t nbytes, uint32_t epoch) {
    pdl_wait();
    const int r = blockIdx.y;
    uint64_t* dst = static_cast<uint64_t*>(p.out[r]);
    const size_t nq = nbytes / 16;
    const size_t q = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (q < nq) {
        const uint4 x = ld_stream(static_cast<const uint4*>(p.in[r]) + q);
        const uint64_t a = make_packet(x.x, epoch), b = make_packet(x.y, epoch);
        const uint64_t c = make_packet(x.z, epoch), d = make_packet(x.w, epoch);
        if (kWide) {
            st_packets4(dst + 4 * q, a, b, c, d);
        } else {
            st_packets2(dst + 4 * q, a, b);
            st_packets2(dst + 4 * q + 2, c, d);
        }
    }
    // Up to 4 packets after the last whole 16 bytes; the last may be padded.
    if (blockIdx.x == 0 && threadIdx.x < 4) {
        const size_t w = 4 * nq + threadIdx.x;
        if (4 * w < nbytes) {
            const uint32_t payload = payload_word(static_cast<const unsigned char*>(p.in[r]), nbytes, w);
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
        st_packet(dst + w, make_packet(payload_word(b, nbytes, w), epoch));
    }
}

// ---------------------------------------------------------------------------
// Poll + unpack + reduce + write-back.  p.in[k] = packet buffer of rank k,
// p.out[j] = output of rank j.  Rank r (blockIdx.y) owns packets
// [r*chunk, min(npk, (r+1)*chunk)), one packet index per thread; vec_out:
// every output is 16-byte aligned, so whole payload words are stored.
// ---------------------------------------------------------------------------
template <int DT, int NR>
__global__ void __launch_bounds__(kThreads)
ll_unpack_reduce_kernel(const RankPtrs p, int n_rt, size_t count, size_t nbytes, size_t chunk, uint32_t epoch,
                        uint64_t max_spins, int32_t* status, bool vec_out) {
    pdl_wait();
    constexpr int EP = PerWord<DT>::kN;
    constexpr int WIN = NR == 0 ? 4 : (NR < 8 ? NR : 8);
    const int n = ranks<NR>(n_rt);
    const size_t npk = (nbytes + 3) / 4;
    const size_t wb = static_cast<size_t>(blockIdx.y) * chunk;
    const size_t w = wb + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (w >= min(npk, wb + chunk)) return;
    float acc[EP];
// Windows of up to 8 ranks: every load of a window is issued before its adds.
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += WIN) {
        uint64_t pk[WIN];
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
            pk[k] = ld_packet(static_cast<const uint64_t*>(p.in[k0 + k]) + w);
        }
#pragma unroll
        for (int k = 0; k < WIN; ++k) {
            if (NR == 0 && k0 + k >= n) break;
            if (!poll_one(static_cast<const uint64_t*>(p.in[k0 + k]) + w, epoch, max_spins, status, pk[k])) return;
            float x[EP];
            widen_word<DT>(packet_payload(pk[k]), x);
#pragma unroll
            for (int e = 0; e < EP; ++e) acc[e] = (k0 + k == 0) ? x[e] : __fadd_rn(acc[e], x[e]);
        }
    }
    if (vec_out && 4 * (w + 1) <= nbytes) {
        const uint32_t y = narrow_word<DT>(acc);
#pragma unroll
        for (int j = 0; j < n; ++j) st_stream_word(static_cast<uint32_t*>(p.out[j]) + w, y);
    } else {
        // Unaligned outputs, or the last payload word holding fewer elements.
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            const size_t i = w * EP + e;
            if (i < count)
                for (int j = 0; j < n; ++j) store_elem<DT>(p.out[j], i, acc[e]);
        }
    }
}

inline unsigned grid_x(size_t items, size_t cap) {
    size_t g = (items + kThreads - 1) / kThreads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

// The byte-wise pack loops over its packets; the vector kernels take one
// item per thread, and a grid they cannot cover is refused.
constexpr size_t kGridCap = 65535;
constexpr size_t kMaxGridX = 0x7FFFFFFF;

template <int DT, int NR>
cudaError_t unpack_dispatch(int nranks, const RankPtrs& p, size_t count, uint32_t epoch, uint64_t max_spins,
                            int32_t* status, bool vec_out, cudaStream_t s) {
    const size_t nbytes = count * Elem<DT>::kSize;
    const size_t npk = (nbytes + 3) / 4;
    const size_t chunk = (npk + nranks - 1) / nranks;
    if ((chunk + kThreads - 1) / kThreads > kMaxGridX) return cudaErrorInvalidValue;
    const dim3 grid(grid_x(chunk, kMaxGridX), nranks);
    launch_kernel(ll_unpack_reduce_kernel<DT, NR>, grid, dim3(kThreads), s, p, nranks, count, nbytes, chunk,
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
        if ((bytes / 16 + kThreads) / kThreads > kMaxGridX) return cudaErrorInvalidValue;
        const dim3 grid(grid_x(bytes / 16 + 1, kMaxGridX), nranks);
        bool wide = true;
        for (int r = 0; r < nranks; ++r) wide = wide && reinterpret_cast<uintptr_t>(p.out[r]) % 32 == 0;
        if (wide) launch_kernel(ll_pack_vec_kernel<true>, grid, dim3(kThreads), stream, p, bytes, epoch);
        else launch_kernel(ll_pack_vec_kernel<false>, grid, dim3(kThreads), stream, p, bytes, epoch);
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
