// convert.cu -- e4m3fn <-> {fp32, fp16, bf16}.
//
// mscclpp commit history (the ROCm FP8 summary and "Add mixed-precision
// accumulation for allreduce"): FP8 data is reduced in a wider type, which
// needs the exact widening e4m3fn -> binary32 and the single saturating
// rounding binary32 -> e4m3fn used inside the reduction kernels.  This entry
// point exposes the same two conversions on their own: dst = R_dst(f32(src)).
// Widening from e4m3fn is exact into every wider type; narrowing rounds once
// to nearest-even with satfinite (finite overflow and infinities -> +-448,
// NaN -> NaN).  Each thread converts 16 elements with 16-byte accesses.
#include "sar_device.cuh"
#include "sar_internal.h"

namespace sar {
namespace {

constexpr int kGroup = 16;   // elements per thread

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
convert_vec_kernel(const void* src, void* dst, size_t count) {
    constexpr int SV = Elem<SRC>::kVE, DV = Elem<DST>::kVE;
    constexpr int SN = kGroup / SV, DN = kGroup / DV;   // 16-byte vectors per group
    const size_t ngroups = count / kGroup;
    for (size_t g = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; g < ngroups;
         g += static_cast<size_t>(gridDim.x) * kThreads) {
        float x[kGroup];
        uint4 in[SN];
#pragma unroll
        for (int m = 0; m < SN; ++m) in[m] = ld_stream(static_cast<const uint4*>(src) + g * SN + m);
#pragma unroll
        for (int m = 0; m < SN; ++m) {
            Acc<SRC> a;
            acc_seed<SRC>(a, in[m]);
#pragma unroll
            for (int e = 0; e < SV; ++e) x[m * SV + e] = a.v[e];
        }
#pragma unroll
        for (int m = 0; m < DN; ++m) {
            Acc<DST> a;
#pragma unroll
            for (int e = 0; e < DV; ++e) a.v[e] = x[m * DV + e];
            st_stream(static_cast<uint4*>(dst) + g * DN + m, acc_round<DST>(a));
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < kGroup) {
        const size_t i = ngroups * kGroup + threadIdx.x;
        if (i < count) store_elem<DST>(dst, i, load_elem<SRC>(src, i));
    }
}

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
convert_scalar_kernel(const void* src, void* dst, size_t count) {
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
        convert_vec_kernel<SRC, DST><<<grid_x(count / kGroup + 1, 0x7FFFFFFF), kThreads, 0, s>>>(src, dst, count);
    } else {
        convert_scalar_kernel<SRC, DST><<<grid_x(count, 16384), kThreads, 0, s>>>(src, dst, count);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_convert(const void* src, sar_dtype src_dt, void* dst, sar_dtype dst_dt, size_t count,
                           bool vec, cudaStream_t stream) {
    if (src_dt == SAR_FP8_E4M3FN) {
        switch (dst_dt) {
        case SAR_FP32: return convert_launch<SAR_FP8_E4M3FN, SAR_FP32>(src, dst, count, vec, stream);
        case SAR_FP16: return convert_launch<SAR_FP8_E4M3FN, SAR_FP16>(src, dst, count, vec, stream);
        case SAR_BF16: return convert_launch<SAR_FP8_E4M3FN, SAR_BF16>(src, dst, count, vec, stream);
        default: break;
        }
    } else if (dst_dt == SAR_FP8_E4M3FN) {
        switch (src_dt) {
        case SAR_FP32: return convert_launch<SAR_FP32, SAR_FP8_E4M3FN>(src, dst, count, vec, stream);
        case SAR_FP16: return convert_launch<SAR_FP16, SAR_FP8_E4M3FN>(src, dst, count, vec, stream);
        case SAR_BF16: return convert_launch<SAR_BF16, SAR_FP8_E4M3FN>(src, dst, count, vec, stream);
        default: break;
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace sar
