// rsag.cu -- the reduce-scatter / all-gather allreduce on one GPU: dispatch
// to the reduce kernels of each element type and accumulator
// (rsag_kernels.cuh, instantiated in rsag_<type>.cu and rsag_<type>_acc.cu)
// and the all-gather broadcast of the two-phase form.
//
// "Support 2 ranks in AllreduceRsAgZeroCopy - #948" ("what changed"): each
// rank reduces its 1/N chunk and writes it back to every peer.  Fused, the
// write-back happens from registers (N*S read + N*S written); in two phases
// the reduce-scatter writes the chunk to the owning rank's output and the
// all-gather copies it from there to every other output: the same N*S
// written, plus one extra S read (the reduced chunks, read back).  That read
// is served by the L2 when the chunks fit there: the reduce-scatter stores
// them with an evict-last policy and the all-gather reads them with
// evict-first.
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

// All-gather: rank r's reduced chunk in out[r] is copied to every other
// output.  One 16-byte load, N-1 stores; one vector per thread, the launch
// covering every whole vector of a chunk (a grid-stride loop kept the N rank
// pointers in registers: 78 registers and 72% of the DRAM peak at 8 ranks).
template <int NR>
__global__ void __launch_bounds__(kThreads)
all_gather_vec_kernel(const RankPtrs p, int n_rt, size_t nbytes, size_t chunk_bytes) {
    pdl_wait();
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk_bytes;
    if (begin >= nbytes) return;
    const size_t end = min(nbytes, begin + chunk_bytes);
    const size_t vbase = begin / 16;
    const size_t nfull = (end - begin) / 16;
    const uint4* src = static_cast<const uint4*>(p.out[r]);
    const size_t v = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (v < nfull) {
        // The reduce-scatter stored this chunk as L2 evict-last; read it
        // from there and let the lines go first from now on.
        const uint4 x = ld_stream_hint(src + vbase + v, l2_policy_evict_first());
#pragma unroll
        for (int j = 0; j < ranks<NR>(n_rt); ++j)
            if (j != r) st_stream(static_cast<uint4*>(p.out[j]) + vbase + v, x);
    }
    // Bytes after the last whole vector (last chunk only).
    if (blockIdx.x == 0 && threadIdx.x < 16) {
        const size_t b = begin + nfull * 16 + threadIdx.x;
        if (b < end) {
            const unsigned char x = static_cast<const unsigned char*>(p.out[r])[b];
#pragma unroll
            for (int j = 0; j < ranks<NR>(n_rt); ++j)
                if (j != r) static_cast<unsigned char*>(p.out[j])[b] = x;
        }
    }
}

template <int NR>
__global__ void __launch_bounds__(kThreads)
all_gather_bytes_kernel(const RankPtrs p, int n_rt, size_t nbytes, size_t chunk_bytes) {
    pdl_wait();
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk_bytes;
    if (begin >= nbytes) return;
    const size_t end = min(nbytes, begin + chunk_bytes);
    const unsigned char* src = static_cast<const unsigned char*>(p.out[r]);
    for (size_t b = begin + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; b < end;
         b += static_cast<size_t>(gridDim.x) * kThreads) {
        const unsigned char x = src[b];
#pragma unroll
        for (int j = 0; j < ranks<NR>(n_rt); ++j)
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

template <int DT>
cudaError_t rsag_typed(RsagMode mode, sar_dtype acc, int nranks, const RankPtrs& p, size_t count, size_t chunk,
                       bool vec, cudaStream_t s) {
    if (acc == SAR_FP32) return launch_rsag_wide<DT>(mode, nranks, p, count, chunk, vec, s);
    if (mode != kFused) return cudaErrorInvalidValue;
    return launch_rsag_narrow<DT>(acc, nranks, p, count, chunk, vec, s);
}

cudaError_t rsag_dispatch(RsagMode mode, sar_dtype acc, sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                          size_t chunk, bool vec, cudaStream_t s) {
    switch (dt) {
    case SAR_BF16: return rsag_typed<SAR_BF16>(mode, acc, nranks, p, count, chunk, vec, s);
    case SAR_FP16: return rsag_typed<SAR_FP16>(mode, acc, nranks, p, count, chunk, vec, s);
    case SAR_FP32: return rsag_typed<SAR_FP32>(mode, acc, nranks, p, count, chunk, vec, s);
    case SAR_FP8_E4M3FN: return rsag_typed<SAR_FP8_E4M3FN>(mode, acc, nranks, p, count, chunk, vec, s);
    case SAR_FP8_E4M3B15: return rsag_typed<SAR_FP8_E4M3B15>(mode, acc, nranks, p, count, chunk, vec, s);
    }
    return cudaErrorInvalidValue;
}

template <int NR>
cudaError_t all_gather_dispatch(const RankPtrs& p, int nranks, size_t nbytes, size_t chunk_bytes, bool vec,
                                cudaStream_t s) {
    if (vec) {
        // one thread per vector: a chunk too large for one grid is refused
        if ((chunk_bytes / 16 + kThreads - 1) / kThreads > kMaxGridX) return cudaErrorInvalidValue;
        const dim3 grid(grid_x(chunk_bytes / 16, kThreads, kMaxGridX), nranks);
        launch_kernel(all_gather_vec_kernel<NR>, grid, dim3(kThreads), s, p, nranks, nbytes,
                      chunk_bytes);
    } else {
        const dim3 grid(grid_x(chunk_bytes, kThreads, kScalarGridX), nranks);
        launch_kernel(all_gather_bytes_kernel<0>, grid, dim3(kThreads), s, p, nranks, nbytes,
                      chunk_bytes);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rsag(RsagMode mode, sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                        size_t chunk, bool vec, cudaStream_t stream) {
    return rsag_dispatch(mode, SAR_FP32, dt, nranks, p, count, chunk, vec, stream);
}

cudaError_t launch_rsag_accum(sar_dtype dt, sar_dtype acc, int nranks, const RankPtrs& p, size_t count,
                              size_t chunk, bool vec, cudaStream_t stream) {
    return rsag_dispatch(kFused, acc, dt, nranks, p, count, chunk, vec, stream);
}

cudaError_t launch_all_gather(int nranks, const RankPtrs& p, size_t count, size_t esize, size_t chunk,
                              bool vec, cudaStream_t stream) {
    const size_t nbytes = count * esize, chunk_bytes = chunk * esize;
    switch (nranks) {
    case 1: return cudaSuccess;   // a single rank already holds its result
    case 2: return all_gather_dispatch<2>(p, 2, nbytes, chunk_bytes, vec, stream);
    case 4: return all_gather_dispatch<4>(p, 4, nbytes, chunk_bytes, vec, stream);
    case 8: return all_gather_dispatch<8>(p, 8, nbytes, chunk_bytes, vec, stream);
    case 16: return all_gather_dispatch<16>(p, 16, nbytes, chunk_bytes, vec, stream);
    case 32: return all_gather_dispatch<32>(p, 32, nbytes, chunk_bytes, vec, stream);
    default:
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        return all_gather_dispatch<0>(p, nranks, nbytes, chunk_bytes, vec, stream);
    }
}

}  // namespace sar
