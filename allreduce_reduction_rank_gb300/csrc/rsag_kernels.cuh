// rsag_kernels.cuh -- the rsag reduce kernels for every accumulator type,
// instantiated per element type by the small rsag_<type>.cu (binary32
// accumulator) and rsag_<type>_acc.cu (narrower accumulators) files.
//
// "Support 2 ranks in AllreduceRsAgZeroCopy - #948" ("what changed"): the rsag
// zero-copy kernel is generic in NRanks, NPeers = NRanks - 1, with the peer
// loops unrolled at compile time; each rank reads its 1/N chunk from every
// peer's input, reduces it and writes it into every peer's output.  Here the
// N ranks are N buffers in this GPU's HBM and rank r is the blockIdx.y slice
// of the grid, so the same structure becomes one streaming kernel:
//
//   per thread and 16-byte vector:  N loads -> sum in rank order -> one
//                                   rounding -> N stores
//
// HBM traffic is the algorithmic minimum, N*S read + N*S written.  NRanks is a
// template parameter, so the rank loops are fully unrolled and every load of
// a tile is issued before the first add.
//
// ACC is the accumulator type (mscclpp commit history, "Add mixed-precision
// accumulation for allreduce": accumDtype).  With ACC = binary32 the partial
// sums are exact binary32 adds; with a narrower ACC every partial sum is
// rounded into ACC: acc_0 = R_acc(x_0), acc_k = R_acc(acc_{k-1} + x_k).
#pragma once

#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace rsag {

// A thread reduces one 16-byte vector per grid-stride step: every rank's
// load of it is issued before the first add (in windows of 8 ranks above 8,
// to bound the registers in flight), and the many small CTAs keep the SMs
// full.  Measured against 2 to 4 vectors per thread: equal or faster at every
// HBM-bound size and up to 30% faster on small calls, where the grid had
// fewer CTAs than SMs.
//
// NR > 0 is a kernel for exactly NR ranks (loops unrolled at compile time);
// NR < 0 is a kernel for at most -NR ranks, the count known only at run time
// (any count up to SAR_MAX_RANKS outside the exact ones), with predicated
// loads: -4 serves 3 ranks, -8 serves 5 to 7 ranks (one window), -32 serves 9
// and more (windows of 4).  A single run-time shape for every count measured
// 85-91% of the copy peak at 3 to 6 ranks.
template <int NR> struct Shape {
    static constexpr int kWin = NR < 8 ? NR : 8;
};
template <> struct Shape<-4> {
    static constexpr int kWin = 4;
};
template <> struct Shape<-8> {
    static constexpr int kWin = 8;
};
template <> struct Shape<-32> {
    static constexpr int kWin = 4;
};

// x -> R_acc(x) as a binary32 value.
template <int ACC> __device__ __forceinline__ float round_acc(float x);
template <> __device__ __forceinline__ float round_acc<SAR_FP32>(float x) { return x; }
template <> __device__ __forceinline__ float round_acc<SAR_FP16>(float x) {
    return __half2float(__float2half_rn(x));
}
template <> __device__ __forceinline__ float round_acc<SAR_BF16>(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}
template <> __device__ __forceinline__ float round_acc<SAR_FP8_E4M3FN>(float x) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3), __NV_E4M3);
    return __half2float(*reinterpret_cast<__half*>(&h));
}

template <> __device__ __forceinline__ float round_acc<SAR_FP8_E4M3B15>(float x) {
    return e4m3b15_to_f32(f32_to_e4m3b15(x));
}

// e4m3b15 with the binary32 accumulator sums 2^8 times the values on the
// e4m3fn conversions (exact, see e4m3b15_widen_scaled); every other vector
// case widens to the values themselves.
template <int DT, int ACC> struct ScaledB15 {
    static constexpr bool k = DT == SAR_FP8_E4M3B15 && ACC == SAR_FP32;
};

// e4m3fn accumulated in e4m3fn ("native") keeps its 16 partial sums as e4m3fn
// values in 8 f16x2 words; a step is one f16x2 add and a round trip through
// the saturating e4m3fn conversion.  This is R(acc + x) exactly: the binary32
// add of two e4m3fn values is exact (multiples of 2^-9 below 2^10), and for
// every one of the 65536 pairs of e4m3fn codes the e4m3fn rounding of their
// binary16 sum equals the e4m3fn rounding of their exact sum (checked
// exhaustively; the binary16 sum is inexact only where the difference cannot
// reach an e4m3fn rounding boundary).
struct AccFn8 { uint32_t h[8]; };

template <int DT, int ACC> struct NativeFn8 {
    static constexpr bool k = DT == SAR_FP8_E4M3FN && ACC == SAR_FP8_E4M3FN;
};

template <int DT, int ACC> struct AccOf { using T = Acc<DT>; };
template <> struct AccOf<SAR_FP8_E4M3FN, SAR_FP8_E4M3FN> { using T = AccFn8; };

// Two e4m3fn codes (low 16 bits) -> their values as f16x2, exactly.
__device__ __forceinline__ uint32_t fn2_to_h2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
// f16x2 -> two e4m3fn codes (low 16 bits): round to nearest even, saturating.
__device__ __forceinline__ uint32_t h2_to_fn2(uint32_t h2) {
    __half2_raw r;
    r.x = static_cast<unsigned short>(h2 & 0xFFFFu);
    r.y = static_cast<unsigned short>(h2 >> 16);
    return __nv_cvt_halfraw2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ uint32_t hadd2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void fn8_seed(AccFn8& a, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a.h[2 * i] = fn2_to_h2(w[i]);
        a.h[2 * i + 1] = fn2_to_h2(w[i] >> 16);
    }
}
__device__ __forceinline__ void fn8_add(AccFn8& a, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a.h[2 * i] = fn2_to_h2(h2_to_fn2(hadd2_rn(a.h[2 * i], fn2_to_h2(w[i]))));
        a.h[2 * i + 1] = fn2_to_h2(h2_to_fn2(hadd2_rn(a.h[2 * i + 1], fn2_to_h2(w[i] >> 16))));
    }
}
__device__ __forceinline__ uint4 fn8_round(const AccFn8& a) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = h2_to_fn2(a.h[2 * i]) | (h2_to_fn2(a.h[2 * i + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT, int ACC> __device__ __forceinline__ void seed(typename AccOf<DT, ACC>::T& a, const uint4& v) {
    if constexpr (NativeFn8<DT, ACC>::k) {
        fn8_seed(a, v);
    } else if constexpr (ScaledB15<DT, ACC>::k) {
        acc_seed_scaled(a, v);
    } else {
        acc_seed<DT>(a, v);
        if constexpr (ACC != SAR_FP32) {
#pragma unroll
            for (int e = 0; e < Elem<DT>::kVE; ++e) a.v[e] = round_acc<ACC>(a.v[e]);
        }
    }
}

template <int DT, int ACC> __device__ __forceinline__ void add(typename AccOf<DT, ACC>::T& a, const uint4& v) {
    if constexpr (NativeFn8<DT, ACC>::k) {
        fn8_add(a, v);
    } else if constexpr (ScaledB15<DT, ACC>::k) {
        acc_add_scaled(a, v);
    } else {
        acc_add<DT>(a, v);
        if constexpr (ACC != SAR_FP32) {
#pragma unroll
            for (int e = 0; e < Elem<DT>::kVE; ++e) a.v[e] = round_acc<ACC>(a.v[e]);
        }
    }
}

template <int DT, int ACC> __device__ __forceinline__ uint4 round_out(const typename AccOf<DT, ACC>::T& a) {
    if constexpr (NativeFn8<DT, ACC>::k) return fn8_round(a);
    else if constexpr (ScaledB15<DT, ACC>::k) return acc_round_scaled(a);
    else return acc_round<DT>(a);
}

// The fused mode writes the result vector to every output.  The reduce-scatter
// mode writes it to the owning rank only, as L2 evict-last, because the
// all-gather step reads it next: two-phase 8 x 64 MiB fp16 went 171.9 ->
// 159.0 us, 2 x 64 MiB bf16 49.3 -> 41.0 us, and results larger than the L2
// (2 x 256 MiB) lost nothing.
template <int MODE, int NR>
__device__ __forceinline__ void store_vector(const RankPtrs& p, int n_rt, int r, size_t v, const uint4& y) {
    if (MODE == kFused) {
#pragma unroll
        for (int j = 0; j < ranks<NR>(n_rt); ++j) st_stream(static_cast<uint4*>(p.out[j]) + v, y);
    } else {
        st_stream_hint(static_cast<uint4*>(p.out[r]) + v, y, l2_policy_evict_last());
    }
}

template <int DT, int NR, int MODE, int ACC>
__device__ __forceinline__ void reduce_element(const RankPtrs& p, int n_rt, int r, size_t i) {
    float acc = round_acc<ACC>(load_elem<DT>(p.in[0], i));
#pragma unroll
    for (int k = 1; k < ranks<NR>(n_rt); ++k) acc = round_acc<ACC>(__fadd_rn(acc, load_elem<DT>(p.in[k], i)));
    if (MODE == kFused) {
#pragma unroll
        for (int j = 0; j < ranks<NR>(n_rt); ++j) store_elem<DT>(p.out[j], i, acc);
    } else {
        store_elem<DT>(p.out[r], i, acc);
    }
}

// A 16-byte vector of -0 codes: -0 is the exact identity of the
// round-to-nearest-even add (x + -0 = x for every x, +0, -0, infinities and
// NaN included), and of a rounding into any accumulator, since an accumulator
// value is representable there.
template <int DT> __device__ __forceinline__ uint4 neg_zero_vec() {
    constexpr uint32_t w = Elem<DT>::kSize == 4 ? 0x80000000u : (Elem<DT>::kSize == 2 ? 0x80008000u : 0x80808080u);
    return make_uint4(w, w, w, w);
}

// Ranks [k0, k0 + WIN) of vector v: loads first, then the in-order adds (the
// first rank seeds the accumulator).  With NR < 0 a rank at or past n_rt is
// not loaded and adds a vector of -0 instead, so the adds need no branches.
template <int DT, int NR, int ACC, int WIN>
__device__ __forceinline__ void reduce_window(const RankPtrs& p, int n_rt, int k0, size_t v,
                                              typename AccOf<DT, ACC>::T& acc) {
    uint4 x[WIN];
#pragma unroll
    for (int k = 0; k < WIN; ++k) {
        const bool live = NR > 0 || k0 + k < n_rt;
        x[k] = live ? ld_stream(static_cast<const uint4*>(p.in[k0 + k]) + v) : neg_zero_vec<DT>();
    }
#pragma unroll
    for (int k = 0; k < WIN; ++k) {
        if (k0 + k == 0) seed<DT, ACC>(acc, x[k]);
        else add<DT, ACC>(acc, x[k]);
    }
}

// One full 16-byte vector (index v counted from the start of the buffers):
// every rank window, one rounding, the stores.  A class whose ranks fit one
// window runs it once at k0 = 0, so its rank pointers are indexed at compile
// time.
template <int DT, int NR, int MODE, int ACC>
__device__ __forceinline__ void reduce_vector(const RankPtrs& p, int n_rt, int r, size_t v) {
    constexpr int WIN = Shape<NR>::kWin;
    typename AccOf<DT, ACC>::T acc;
    if constexpr (NR < 0 && -NR <= WIN) {
        reduce_window<DT, NR, ACC, WIN>(p, n_rt, 0, v, acc);
    } else {
#pragma unroll 1
        for (int k0 = 0; k0 < ranks<NR>(n_rt); k0 += WIN) reduce_window<DT, NR, ACC, WIN>(p, n_rt, k0, v, acc);
    }
    store_vector<MODE, NR>(p, n_rt, r, v, round_out<DT, ACC>(acc));
}

// Vector kernel: grid = (CTAs over chunk r, nranks), one vector per thread;
// the launch covers every vector of a chunk.  Requires every buffer to be
// 16-byte aligned; chunk is a multiple of the vector length, so only the last
// chunk can end inside a vector, and that partial vector is reduced element
// by element.
// BT: threads per CTA (kThreads, or kSmallThreads for small calls).
template <int DT, int NR, int MODE, int ACC, int BT>
__global__ void __launch_bounds__(BT)
vec_kernel(const RankPtrs p, int n_rt, size_t count, size_t chunk) {
    pdl_wait();
    constexpr int VE = Elem<DT>::kVE;
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk;
    if (begin >= count) return;
    const size_t end = min(count, begin + chunk);
    const size_t vbase = begin / VE;
    const size_t nfull = (end - begin) / VE;            // whole vectors in the chunk
    const size_t nvec = (end - begin + VE - 1) / VE;    // plus a partial one at the very end
    const size_t v = static_cast<size_t>(blockIdx.x) * BT + threadIdx.x;
    if (v < nfull) {
        reduce_vector<DT, NR, MODE, ACC>(p, n_rt, r, vbase + v);
    } else if (v < nvec) {
        for (size_t i = begin + v * VE; i < end; ++i) reduce_element<DT, NR, MODE, ACC>(p, n_rt, r, i);
    }
}

// Element kernel for buffers that are not all 16-byte aligned (the slow
// path): the rank loop runs to the runtime nranks, so one instantiation
// serves every rank count.
template <int DT, int MODE, int ACC>
__global__ void __launch_bounds__(kThreads)
scalar_kernel(const RankPtrs p, int nranks, size_t count, size_t chunk) {
    pdl_wait();
    const int r = blockIdx.y;
    const size_t begin = static_cast<size_t>(r) * chunk;
    if (begin >= count) return;
    const size_t end = min(count, begin + chunk);
    for (size_t i = begin + static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < end;
         i += static_cast<size_t>(gridDim.x) * kThreads)
        reduce_element<DT, 0, MODE, ACC>(p, nranks, r, i);
}

inline unsigned grid_x(size_t items, size_t per_cta, size_t cap) {
    size_t g = (items + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

constexpr size_t kMaxGridX = 0x7FFFFFFF;
constexpr size_t kScalarGridX = 8192;

// Calls whose grid of 256-thread CTAs would hold fewer than kSmallGridCtas
// CTAs over all ranks run CTAs of kSmallThreads instead, twice as many of
// them, on more SMs.  Measured on GB300 (2 ranks bf16, CUDA graph, us per
// call, 256 / 128 threads): 16 KiB 1.086 / 1.002, 64 KiB 1.173 / 1.086,
// 256 KiB 1.198 / 1.163, 1 MiB 1.419 / 1.405, 4 MiB 2.350 / 2.387.
constexpr int kSmallThreads = 128;
constexpr size_t kSmallGridCtas = 256;

// The fused kernels for more than 8 ranks (16 and 32, and the run-time class
// up to 32) run CTAs of kManyRankThreads at every size: with that launch
// bound the compiler keeps two windows of rank loads in flight instead of one
// (72 registers instead of 40 at 32 ranks).  Measured on GB300 (fp32, CUDA
// graph, us per call, 256 or 128 / 32 threads): 16 x 64 KiB 2.21 / 1.55,
// 32 x 64 KiB 3.55 / 2.31, 16 x 1 MiB 4.66 / 4.25, 32 x 1 MiB 7.79 / 7.33,
// 12 x 64 KiB 2.19 / 1.99; 16 x 32 MiB, 32 x 8 MiB and 12 x 64 MiB fp16
// unchanged.  The reduce-scatter kernel keeps its CTAs (32 x 8 MiB fp32
// two-phase was 1.3% slower with 32 threads).
constexpr int kManyRankThreads = 32;

template <int DT, int NR, int MODE, int ACC>
cudaError_t launch_vec(const RankPtrs& p, int nranks, size_t count, size_t chunk, cudaStream_t s) {
    constexpr int VE = Elem<DT>::kVE;
    // one thread per vector of a chunk: a chunk too large for one grid (over
    // 2^31 CTAs of 256 vectors, 8 TiB per rank) is refused, never cut short
    const size_t vecs = (chunk + VE - 1) / VE;
    const size_t ctas = (vecs + kThreads - 1) / kThreads;
    if (ctas > kMaxGridX) return cudaErrorInvalidValue;
    if constexpr (MODE == kFused && (NR > 8 || NR == -32)) {
        if ((vecs + kManyRankThreads - 1) / kManyRankThreads <= kMaxGridX) {
            const dim3 grid(grid_x(vecs, kManyRankThreads, kMaxGridX), nranks);
            launch_kernel(vec_kernel<DT, NR, MODE, ACC, kManyRankThreads>, grid, dim3(kManyRankThreads), s, p,
                          nranks, count, chunk);
            return cudaGetLastError();
        }
    }
    if (ctas * static_cast<size_t>(nranks) < kSmallGridCtas) {
        const dim3 grid(grid_x(vecs, kSmallThreads, kMaxGridX), nranks);
        launch_kernel(vec_kernel<DT, NR, MODE, ACC, kSmallThreads>, grid, dim3(kSmallThreads), s, p, nranks, count,
                      chunk);
    } else {
        const dim3 grid(grid_x(vecs, kThreads, kMaxGridX), nranks);
        launch_kernel(vec_kernel<DT, NR, MODE, ACC, kThreads>, grid, dim3(kThreads), s, p, nranks, count, chunk);
    }
    return cudaGetLastError();
}

template <int DT, int MODE, int ACC>
cudaError_t launch_ranks(int nranks, const RankPtrs& p, size_t count, size_t chunk, bool vec, cudaStream_t s) {
    if (!vec) {
        const dim3 grid(grid_x(chunk, kThreads, kScalarGridX), nranks);
            launch_kernel(scalar_kernel<DT, MODE, ACC>, grid, dim3(kThreads), s, p, nranks, count, chunk);
        return cudaGetLastError();
    }
    switch (nranks) {
    case 1: return launch_vec<DT, 1, MODE, ACC>(p, 1, count, chunk, s);
    case 2: return launch_vec<DT, 2, MODE, ACC>(p, 2, count, chunk, s);
    case 4: return launch_vec<DT, 4, MODE, ACC>(p, 4, count, chunk, s);
    case 8: return launch_vec<DT, 8, MODE, ACC>(p, 8, count, chunk, s);
    case 16: return launch_vec<DT, 16, MODE, ACC>(p, 16, count, chunk, s);
    case 32: return launch_vec<DT, 32, MODE, ACC>(p, 32, count, chunk, s);
    default:
        // any other count: a kernel for the smallest class that holds it
        if (nranks < 1 || nranks > SAR_MAX_RANKS) return cudaErrorInvalidValue;
        if (nranks <= 4) return launch_vec<DT, -4, MODE, ACC>(p, nranks, count, chunk, s);
        if (nranks <= 8) return launch_vec<DT, -8, MODE, ACC>(p, nranks, count, chunk, s);
        return launch_vec<DT, -32, MODE, ACC>(p, nranks, count, chunk, s);
    }
}

}  // namespace rsag

// The reduce launchers of one element type: binary32 accumulation in either
// mode (instantiated in rsag_<type>.cu), and fp16, bf16 or, for FP8 types,
// native accumulation in the fused mode (instantiated in rsag_<type>_acc.cu).
template <int DT>
cudaError_t launch_rsag_wide(RsagMode mode, int nranks, const RankPtrs& p, size_t count, size_t chunk, bool vec,
                             cudaStream_t s) {
    if (mode == kFused) return rsag::launch_ranks<DT, kFused, SAR_FP32>(nranks, p, count, chunk, vec, s);
    return rsag::launch_ranks<DT, kReduceScatter, SAR_FP32>(nranks, p, count, chunk, vec, s);
}

template <int DT>
cudaError_t launch_rsag_narrow(sar_dtype acc, int nranks, const RankPtrs& p, size_t count, size_t chunk, bool vec,
                               cudaStream_t s) {
    switch (acc) {
    case SAR_FP16: return rsag::launch_ranks<DT, kFused, SAR_FP16>(nranks, p, count, chunk, vec, s);
    case SAR_BF16: return rsag::launch_ranks<DT, kFused, SAR_BF16>(nranks, p, count, chunk, vec, s);
    case SAR_FP8_E4M3FN:
        if constexpr (DT == SAR_FP8_E4M3FN)
            return rsag::launch_ranks<DT, kFused, SAR_FP8_E4M3FN>(nranks, p, count, chunk, vec, s);
        return cudaErrorInvalidValue;
    case SAR_FP8_E4M3B15:
        if constexpr (DT == SAR_FP8_E4M3B15)
            return rsag::launch_ranks<DT, kFused, SAR_FP8_E4M3B15>(nranks, p, count, chunk, vec, s);
        return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sar
