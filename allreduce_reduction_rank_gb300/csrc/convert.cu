// convert.cu -- FP8 (e4m3fn, e4m3b15) <-> {fp32, fp16, bf16}.
//
// mscclpp commit history (the ROCm FP8 summary, "Add fp8_e4m3b15 datatype"
// and "Add mixed-precision accumulation for allreduce"): FP8 data is reduced
// in a wider type, which needs the exact widening FP8 -> binary32 and the
// single rounding binary32 -> FP8 used inside the reduction kernels.  This
// entry point exposes the same conversions on their own: dst = R_dst(f32(src)).
// Widening is exact into every wider type; narrowing rounds once to
// nearest-even (e4m3fn: satfinite, finite overflow and infinities -> +-448;
// e4m3b15: overflow -> infinity; NaN -> NaN).  Each lane converts 4
// consecutive elements per access, so a warp's loads and stores each cover
// one contiguous run of memory.
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

// A quad is 4 consecutive elements: 4, 8 or 16 bytes depending on the type.
// Lane l of a warp handles quad base + 32*u + l for u = 0..kUnroll-1, so every
// warp-wide load and store covers one contiguous run of memory.
constexpr int kUnroll = 4;

template <int DT> __device__ __forceinline__ void quad_load(const void* base, size_t q, float (&x)[4]);
template <int DT> __device__ __forceinline__ void quad_store(void* base, size_t q, const float (&x)[4]);

template <int DT> __device__ __forceinline__ void quad_load8(const void* base, size_t q, float (&x)[4]) {
    uint32_t w;
    asm("ld.global.L1::no_allocate.u32 %0, [%1];" : "=r"(w) : "l"(static_cast<const uint32_t*>(base) + q));
    widen_word<DT>(w, x);
}
template <> __device__ __forceinline__ void quad_load<SAR_FP8_E4M3FN>(const void* base, size_t q, float (&x)[4]) {
    quad_load8<SAR_FP8_E4M3FN>(base, q, x);
}
template <> __device__ __forceinline__ void quad_load<SAR_FP8_E4M3B15>(const void* base, size_t q, float (&x)[4]) {
    quad_load8<SAR_FP8_E4M3B15>(base, q, x);
}
template <int DT> __device__ __forceinline__ void quad_load16(const void* base, size_t q, float (&x)[4]) {
    uint32_t a, b;
    asm("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
        : "=r"(a), "=r"(b)
        : "l"(static_cast<const uint2*>(base) + q));
    widen_word<DT>(a, x);
    widen_word<DT>(b, x + 2);
}
template <> __device__ __forceinline__ void quad_load<SAR_FP16>(const void* base, size_t q, float (&x)[4]) {
    quad_load16<SAR_FP16>(base, q, x);
}
template <> __device__ __forceinline__ void quad_load<SAR_BF16>(const void* base, size_t q, float (&x)[4]) {
    quad_load16<SAR_BF16>(base, q, x);
}
template <> __device__ __forceinline__ void quad_load<SAR_FP32>(const void* base, size_t q, float (&x)[4]) {
    const uint4 v = ld_stream(static_cast<const uint4*>(base) + q);
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}

template <int DT> __device__ __forceinline__ void quad_store8(void* base, size_t q, const float (&x)[4]) {
    const uint32_t w = narrow_word<DT>(x);
    asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" :: "l"(static_cast<uint32_t*>(base) + q), "r"(w)
                 : "memory");
}
template <> __device__ __forceinline__ void quad_store<SAR_FP8_E4M3FN>(void* base, size_t q, const float (&x)[4]) {
    quad_store8<SAR_FP8_E4M3FN>(base, q, x);
}
template <> __device__ __forceinline__ void quad_store<SAR_FP8_E4M3B15>(void* base, size_t q, const float (&x)[4]) {
    quad_store8<SAR_FP8_E4M3B15>(base, q, x);
}
template <int DT> __device__ __forceinline__ void quad_store16(void* base, size_t q, const float (&x)[4]) {
    const uint32_t a = narrow_word<DT>(x), b = narrow_word<DT>(x + 2);
    asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1, %2};" :: "l"(static_cast<uint2*>(base) + q),
                 "r"(a), "r"(b) : "memory");
}
template <> __device__ __forceinline__ void quad_store<SAR_FP16>(void* base, size_t q, const float (&x)[4]) {
    quad_store16<SAR_FP16>(base, q, x);
}
template <> __device__ __forceinline__ void quad_store<SAR_BF16>(void* base, size_t q, const float (&x)[4]) {
    quad_store16<SAR_BF16>(base, q, x);
}
template <> __device__ __forceinline__ void quad_store<SAR_FP32>(void* base, size_t q, const float (&x)[4]) {
    st_stream(static_cast<uint4*>(base) + q,
              make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3])));
}

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
convert_vec_kernel(const void* src, void* dst, size_t count) {
    pdl_wait();
    const size_t nq = count / 4;
    const unsigned lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t base = warp * 32 * kUnroll; base < nq; base += nwarps * 32 * kUnroll) {
        float x[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t q = base + 32 * u + lane;
            if (q < nq) quad_load<SRC>(src, q, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const size_t q = base + 32 * u + lane;
            if (q < nq) quad_store<DST>(dst, q, x[u]);
        }
    }
    // The last count % 4 elements.
    if (blockIdx.x == 0 && threadIdx.x < 4) {
        const size_t i = nq * 4 + threadIdx.x;
        if (i < count) store_elem<DST>(dst, i, load_elem<SRC>(src, i));
    }
}

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
convert_scalar_kernel(const void* src, void* dst, size_t count) {
    pdl_wait();
    for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < count;
         i += static_cast<size_t>(gridDim.x) * kThreads)
        store_elem<DST>(dst, i, load_elem<SRC>(src, i));
}

inline unsigned grid_x(size_t items, size_t cap) {
    size_t g = (items + kThreads - 1) / kThreads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return static_cast<unsigned>(g);
}

template <int SRC, int DST>
cudaError_t convert_launch(const void* src, void* dst, size_t count, bool vec, cudaStream_t s) {
    if (vec) {
        // one warp per 32 * kUnroll quads
        const size_t warps = (count / 4 + 32 * kUnroll - 1) / (32 * kUnroll);
        launch_kernel(convert_vec_kernel<SRC, DST>, dim3(grid_x(warps * 32 + 1, 0x7FFFFFFF)),
                      dim3(kThreads), s, src, dst, count);
    } else {
        launch_kernel(convert_scalar_kernel<SRC, DST>, dim3(grid_x(count, 16384)), dim3(kThreads), s,
                      src, dst, count);
    }
    return cudaGetLastError();
}

}  // namespace

template <int FP8>
cudaError_t convert_fp8_pairs(const void* src, sar_dtype src_dt, void* dst, sar_dtype dst_dt, size_t count,
                              bool vec, cudaStream_t stream) {
    if (src_dt == FP8) {
        switch (dst_dt) {
        case SAR_FP32: return convert_launch<FP8, SAR_FP32>(src, dst, count, vec, stream);
        case SAR_FP16: return convert_launch<FP8, SAR_FP16>(src, dst, count, vec, stream);
        case SAR_BF16: return convert_launch<FP8, SAR_BF16>(src, dst, count, vec, stream);
        default: break;
        }
    } else if (dst_dt == FP8) {
        switch (src_dt) {
        case SAR_FP32: return convert_launch<SAR_FP32, FP8>(src, dst, count, vec, stream);
        case SAR_FP16: return convert_launch<SAR_FP16, FP8>(src, dst, count, vec, stream);
        case SAR_BF16: return convert_launch<SAR_BF16, FP8>(src, dst, count, vec, stream);
        default: break;
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_convert(const void* src, sar_dtype src_dt, void* dst, sar_dtype dst_dt, size_t count,
                           bool vec, cudaStream_t stream) {
    if (src_dt == SAR_FP8_E4M3FN || dst_dt == SAR_FP8_E4M3FN)
        return convert_fp8_pairs<SAR_FP8_E4M3FN>(src, src_dt, dst, dst_dt, count, vec, stream);
    return convert_fp8_pairs<SAR_FP8_E4M3B15>(src, src_dt, dst, dst_dt, count, vec, stream);
}

}  // namespace sar
