// rsag.cu -- the reduce-scatter / all-gather allreduce on one GPU.
//
// "Support 2 ranks in AllreduceRsAgZeroCopy - #948" ("what changed"): the rsag
// zero-copy kernel is generic in NRanks, NPeers = NRanks - 1, with the peer
// loops unrolled at compile time; each rank reads its 1/N chunk from every
// peer's input, reduces it and writes it into every peer's output.  Here the
// N ranks are N buffers in this GPU's HBM and rank r is the blockIdx.y slice
// of the grid, so the same structure becomes one streaming kernel:
//
//   per thread and 16-byte vector:  N loads -> binary32 sum in rank order
//                                   -> one rounding -> N stores
//
// HBM traffic is the algorithmic minimum, N*S read + N*S written.  NRanks is a
// template parameter, so the rank loops are fully unrolled and every load of
// a tile is issued before the first add.
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

// Loads in flight per thread: all ranks for up to 8 ranks (x UNROLL vectors),
// windows of 8 ranks above that to bound register use.
template <int NR> struct RsagShape {
    static constexpr int kWin = NR < 8 ? NR : 8;
    static constexpr int kUnroll = NR <= 2 ? 4 : (NR <= 8 ? 2 : 1);
};

template <int MODE, int NR>
__device__ __forceinline__ void store_vector(const RankPtrs& p, int r, size_t v, const uint4& y) {
    if (MODE == kFused) {
#pragma unroll
        for (int j = 0; j < NR; ++j) st_stream(static_cast<uint4*>(p.out[j]) + v, y);
    } else {
        st_stream(static_cast<uint4*>(p.out[r]) + v, y);
    }
}

template <int DT, int NR, int MODE>
__device__ __forceinline__ void reduce_element(const RankPtrs& p, int r, size_t i) {
    float acc = load_elem<DT>(p.in[0], i);
#pragma unroll
    for (int k = 1; k < NR; ++k) acc = __fadd_rn(acc, load_elem<DT>(p.in[k], i));
    if (MODE == kFused) {
#pragma unroll
        for (int j = 0; j < NR; ++j) store_elem<DT>(p.out[j], i, acc);
    } else {
        store_elem<DT>(p.out[r], i, acc);
    }
}

// One full 16-byte vector (index v counted from the start of the buffers).
template <int DT, int NR, int MODE>
__device__ __forceinline__ void reduce_vector(const RankPtrs& p, int r, size_t v) {
    Acc<DT> acc;
    uint4 x[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) x[k] = ld_stream(static_cast<const uint4*>(p.in[k]) + v);
    acc_seed<DT>(acc, x[0]);
#pragma unroll
    for (int k = 1; k < NR; ++k) acc_add<DT>(acc, x[k]);
    store_vector<MODE, NR>(p, r, v, acc_round<DT>(acc));
}

// Vector kernel: grid = (tiles of chunk r, nranks).  Requires every buffer to
// be 16-byte aligned; chunk is a multiple of the vector length.
template <int DT, int NR, int MODE>
__global__ void __launch_bounds__(kThreads)
rsag_vec_kernel(const RankPtrs p, size_t count, size_t chunk) {
    constexpr int VE = Elem<DT>::kVE;
    constexpr int WIN = RsagShape<NR>::kWin;
    constexpr int UNROLL = RsagShape<NR>::kUnroll;
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk;
    if (begin >= count) return;
    const size_t end = min(count, begin + chunk);
    const size_t vbase = begin / VE;
    const size_t nfull = (end - begin) / VE;            // whole vectors in the chunk
    const size_t nvec = (end - begin + VE - 1) / VE;    // plus a partial one at the very end
    const size_t tile = static_cast<size_t>(kThreads) * UNROLL;

    for (size_t t0 = static_cast<size_t>(blockIdx.x) * tile; t0 < nvec;
         t0 += static_cast<size_t>(gridDim.x) * tile) {
        if (t0 + tile <= nfull) {
            // Interior tile: UNROLL vectors per thread, all loads of a rank
            // window issued before the first add.
            Acc<DT> acc[UNROLL];
#pragma unroll
            for (int k0 = 0; k0 < NR; k0 += WIN) {
                uint4 x[WIN][UNROLL];
#pragma unroll
                for (int k = 0; k < WIN; ++k)
#pragma unroll
                    for (int u = 0; u < UNROLL; ++u)
                        x[k][u] = ld_stream(static_cast<const uint4*>(p.in[k0 + k]) + vbase + t0 +
                                            u * kThreads + threadIdx.x);
#pragma unroll
                for (int k = 0; k < WIN; ++k)
#pragma unroll
                    for (int u = 0; u < UNROLL; ++u) {
                        if (k0 + k == 0) acc_seed<DT>(acc[u], x[k][u]);
                        else acc_add<DT>(acc[u], x[k][u]);
                    }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                store_vector<MODE, NR>(p, r, vbase + t0 + u * kThreads + threadIdx.x,
                                       acc_round<DT>(acc[u]));
        } else {
            // Edge tile: whole vectors one at a time, then the partial vector
            // (only the last chunk can end inside a vector) element by element.
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const size_t v = t0 + u * kThreads + threadIdx.x;
                if (v < nfull) {
                    reduce_vector<DT, NR, MODE>(p, r, vbase + v);
                } else if (v < nvec) {
                    for (size_t i = begin + v * VE; i < end; ++i) reduce_element<DT, NR, MODE>(p, r, i);
                }
            }
        }
    }
}

// Element kernel for buffers that are not all 16-byte aligned.
template <int DT, int NR, int MODE>
__global__ void __launch_bounds__(kThreads)
rsag_scalar_kernel(const RankPtrs p, size_t count, size_t chunk) {
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk;
    if (begin >= count) return;
    const size_t end = min(count, begin + chunk);
    for (size_t i = begin + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < end;
         i += static_cast<size_t>(gridDim.x) * kThreads)
        reduce_element<DT, NR, MODE>(p, r, i);
}

// All-gather: rank r's reduced chunk in out[r] is copied to every other
// output.  One 16-byte load, N-1 stores.
template <int NR>
__global__ void __launch_bounds__(kThreads)
all_gather_vec_kernel(const RankPtrs p, size_t nbytes, size_t chunk_bytes) {
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk_bytes;
    if (begin >= nbytes) return;
    const size_t end = min(nbytes, begin + chunk_bytes);
    const size_t vbase = begin / 16;
    const size_t nfull = (end - begin) / 16;
    const uint4* src = static_cast<const uint4*>(p.out[r]);
    for (size_t v = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; v < nfull;
         v += static_cast<size_t>(gridDim.x) * kThreads) {
        const uint4 x = ld_stream(src + vbase + v);
#pragma unroll
        for (int j = 0; j < NR; ++j)
            if (j != r) st_stream(static_cast<uint4*>(p.out[j]) + vbase + v, x);
    }
    // Bytes after the last whole vector (last chunk only).
    if (blockIdx.x == 0 && threadIdx.x < 16) {
        const size_t b = begin + nfull * 16 + threadIdx.x;
        if (b < end) {
            const unsigned char x = static_cast<const unsigned char*>(p.out[r])[b];
#pragma unroll
            for (int j = 0; j < NR; ++j)
                if (j != r) static_cast<unsigned char*>(p.out[j])[b] = x;
        }
    }
}

template <int NR>
__global__ void __launch_bounds__(kThreads)
all_gather_bytes_kernel(const RankPtrs p, size_t nbytes, size_t chunk_bytes) {
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk_bytes;
    if (begin >= nbytes) return;
    const size_t end = min(nbytes, begin + chunk_bytes);
    const unsigned char* src = static_cast<const unsigned char*>(p.out[r]);
    for (size_t b = begin + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; b < end;
         b += static_cast<size_t>(gridDim.x) * kThreads) {
        const unsigned char x = src[b];
#pragma unroll
        for (int j = 0; j < NR; ++j)
            if (j != r) static_cast<unsigned char*>(p.out[j])[b] = x;
    }
}

inline unsigned grid_x(size_t items, size_t per_cta, size_t cap) {
    size_t g = (items + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

constexpr size_t kMaxGridX = 0x7FFFFFFF;
constexpr size_t kScalarGridX = 8192;

template <int DT, int NR>
cudaError_t rsag_dispatch_mode(RsagMode mode, const RankPtrs& p, size_t count, size_t chunk, bool vec,
                               cudaStream_t s) {
    constexpr int VE = Elem<DT>::kVE;
    if (vec) {
        const size_t tile = static_cast<size_t>(kThreads) * RsagShape<NR>::kUnroll;
        const dim3 grid(grid_x((chunk + VE - 1) / VE, tile, kMaxGridX), NR);
        if (mode == kFused) rsag_vec_kernel<DT, NR, kFused><<<grid, kThreads, 0, s>>>(p, count, chunk);
        else rsag_vec_kernel<DT, NR, kReduceScatter><<<grid, kThreads, 0, s>>>(p, count, chunk);
    } else {
        const dim3 grid(grid_x(chunk, kThreads, kScalarGridX), NR);
        if (mode == kFused) rsag_scalar_kernel<DT, NR, kFused><<<grid, kThreads, 0, s>>>(p, count, chunk);
        else rsag_scalar_kernel<DT, NR, kReduceScatter><<<grid, kThreads, 0, s>>>(p, count, chunk);
    }
    return cudaGetLastError();
}

template <int DT>
cudaError_t rsag_dispatch_ranks(RsagMode mode, int nranks, const RankPtrs& p, size_t count, size_t chunk,
                                bool vec, cudaStream_t s) {
    switch (nranks) {
    case 1: return rsag_dispatch_mode<DT, 1>(mode, p, count, chunk, vec, s);
    case 2: return rsag_dispatch_mode<DT, 2>(mode, p, count, chunk, vec, s);
    case 4: return rsag_dispatch_mode<DT, 4>(mode, p, count, chunk, vec, s);
    case 8: return rsag_dispatch_mode<DT, 8>(mode, p, count, chunk, vec, s);
    case 16: return rsag_dispatch_mode<DT, 16>(mode, p, count, chunk, vec, s);
    case 32: return rsag_dispatch_mode<DT, 32>(mode, p, count, chunk, vec, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int NR>
cudaError_t all_gather_dispatch(const RankPtrs& p, size_t nbytes, size_t chunk_bytes, bool vec,
                                cudaStream_t s) {
    if (vec) {
        const dim3 grid(grid_x(chunk_bytes / 16, kThreads, kMaxGridX), NR);
        all_gather_vec_kernel<NR><<<grid, kThreads, 0, s>>>(p, nbytes, chunk_bytes);
    } else {
        const dim3 grid(grid_x(chunk_bytes, kThreads, kScalarGridX), NR);
        all_gather_bytes_kernel<NR><<<grid, kThreads, 0, s>>>(p, nbytes, chunk_bytes);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rsag(RsagMode mode, sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                        size_t chunk, bool vec, cudaStream_t stream) {
    switch (dt) {
    case SAR_BF16: return rsag_dispatch_ranks<SAR_BF16>(mode, nranks, p, count, chunk, vec, stream);
    case SAR_FP16: return rsag_dispatch_ranks<SAR_FP16>(mode, nranks, p, count, chunk, vec, stream);
    case SAR_FP32: return rsag_dispatch_ranks<SAR_FP32>(mode, nranks, p, count, chunk, vec, stream);
    case SAR_FP8_E4M3FN:
        return rsag_dispatch_ranks<SAR_FP8_E4M3FN>(mode, nranks, p, count, chunk, vec, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_all_gather(int nranks, const RankPtrs& p, size_t count, size_t esize, size_t chunk,
                              bool vec, cudaStream_t stream) {
    const size_t nbytes = count * esize, chunk_bytes = chunk * esize;
    switch (nranks) {
    case 1: return cudaSuccess;   // a single rank already holds its result
    case 2: return all_gather_dispatch<2>(p, nbytes, chunk_bytes, vec, stream);
    case 4: return all_gather_dispatch<4>(p, nbytes, chunk_bytes, vec, stream);
    case 8: return all_gather_dispatch<8>(p, nbytes, chunk_bytes, vec, stream);
    case 16: return all_gather_dispatch<16>(p, nbytes, chunk_bytes, vec, stream);
    case 32: return all_gather_dispatch<32>(p, nbytes, chunk_bytes, vec, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sar
