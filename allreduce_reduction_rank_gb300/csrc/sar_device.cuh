// sar_device.cuh -- element types, 16-byte vector I/O and the in-order
// binary32 accumulation shared by the rsag and LL kernels.
//
// Arithmetic contract (mscclpp commit history, "Add mixed-precision
// accumulation for allreduce": FP8/16-bit inputs reduced in float32): every
// element is widened exactly to binary32, the ranks are added in order
// 0..N-1 with IEEE round-to-nearest-even adds (__fadd_rn: never contracted,
// never flushed; this library is built without fast-math or ftz), and the sum
// is rounded once to the element type with the hardware cvt.rn conversions
// (satfinite for e4m3fn).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/sar.h"

namespace sar {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// Element types.  kVE = elements per 16-byte vector.
// ---------------------------------------------------------------------------
template <int DT> struct Elem;
template <> struct Elem<SAR_BF16> { static constexpr int kSize = 2, kVE = 8; };
template <> struct Elem<SAR_FP16> { static constexpr int kSize = 2, kVE = 8; };
template <> struct Elem<SAR_FP32> { static constexpr int kSize = 4, kVE = 4; };
template <> struct Elem<SAR_FP8_E4M3FN> { static constexpr int kSize = 1, kVE = 16; };

// Exact widening of one 32-bit word holding 2 (16-bit types), 1 (fp32) or
// 4 (e4m3fn) elements, lowest address first.
template <int DT> __device__ __forceinline__ void widen_word(uint32_t w, float* x);

template <> __device__ __forceinline__ void widen_word<SAR_BF16>(uint32_t w, float* x) {
    x[0] = __uint_as_float(w << 16);          // bfloat16 is the top half of a binary32
    x[1] = __uint_as_float(w & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void widen_word<SAR_FP16>(uint32_t w, float* x) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    x[0] = f.x;
    x[1] = f.y;
}
template <> __device__ __forceinline__ void widen_word<SAR_FP32>(uint32_t w, float* x) {
    x[0] = __uint_as_float(w);
}
template <> __device__ __forceinline__ void widen_word<SAR_FP8_E4M3FN>(uint32_t w, float* x) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
    float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// One rounding of binary32 values into a 32-bit word of elements.
template <int DT> __device__ __forceinline__ uint32_t narrow_word(const float* x);

template <> __device__ __forceinline__ uint32_t narrow_word<SAR_BF16>(const float* x) {
    __nv_bfloat162 v = __floats2bfloat162_rn(x[0], x[1]);
    return *reinterpret_cast<uint32_t*>(&v);
}
template <> __device__ __forceinline__ uint32_t narrow_word<SAR_FP16>(const float* x) {
    __half2 v = __floats2half2_rn(x[0], x[1]);
    return *reinterpret_cast<uint32_t*>(&v);
}
template <> __device__ __forceinline__ uint32_t narrow_word<SAR_FP32>(const float* x) {
    return __float_as_uint(x[0]);
}
template <> __device__ __forceinline__ uint32_t narrow_word<SAR_FP8_E4M3FN>(const float* x) {
    uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
    uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[2], x[3]), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}

// Elements per 32-bit word.
template <int DT> struct PerWord { static constexpr int kN = 4 / Elem<DT>::kSize; };

// ---------------------------------------------------------------------------
// 16-byte vectors.
// ---------------------------------------------------------------------------
template <int DT> struct Acc { float v[Elem<DT>::kVE]; };

// acc = f32(v) (the seed: rank 0's element, not 0 + element, so that a single
// rank is the identity and -0 stays -0).
template <int DT> __device__ __forceinline__ void acc_seed(Acc<DT>& a, const uint4& v) {
    constexpr int W = PerWord<DT>::kN;
    widen_word<DT>(v.x, a.v + 0 * W);
    widen_word<DT>(v.y, a.v + 1 * W);
    widen_word<DT>(v.z, a.v + 2 * W);
    widen_word<DT>(v.w, a.v + 3 * W);
}

// acc += f32(v), one binary32 add per element.
template <int DT> __device__ __forceinline__ void acc_add(Acc<DT>& a, const uint4& v) {
    constexpr int W = PerWord<DT>::kN;
    float x[Elem<DT>::kVE];
    widen_word<DT>(v.x, x + 0 * W);
    widen_word<DT>(v.y, x + 1 * W);
    widen_word<DT>(v.z, x + 2 * W);
    widen_word<DT>(v.w, x + 3 * W);
#pragma unroll
    for (int e = 0; e < Elem<DT>::kVE; ++e) a.v[e] = __fadd_rn(a.v[e], x[e]);
}

template <int DT> __device__ __forceinline__ uint4 acc_round(const Acc<DT>& a) {
    constexpr int W = PerWord<DT>::kN;
    uint4 r;
    r.x = narrow_word<DT>(a.v + 0 * W);
    r.y = narrow_word<DT>(a.v + 1 * W);
    r.z = narrow_word<DT>(a.v + 2 * W);
    r.w = narrow_word<DT>(a.v + 3 * W);
    return r;
}

// ---------------------------------------------------------------------------
// Scalar element access (tails and unaligned buffers).
// ---------------------------------------------------------------------------
template <int DT> __device__ __forceinline__ float load_elem(const void* base, size_t i);
template <> __device__ __forceinline__ float load_elem<SAR_BF16>(const void* base, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[i]) << 16);
}
template <> __device__ __forceinline__ float load_elem<SAR_FP16>(const void* base, size_t i) {
    return __half2float(static_cast<const __half*>(base)[i]);
}
template <> __device__ __forceinline__ float load_elem<SAR_FP32>(const void* base, size_t i) {
    return static_cast<const float*>(base)[i];
}
template <> __device__ __forceinline__ float load_elem<SAR_FP8_E4M3FN>(const void* base, size_t i) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<const __nv_fp8_storage_t*>(base)[i], __NV_E4M3);
    return __half2float(*reinterpret_cast<__half*>(&h));
}

template <int DT> __device__ __forceinline__ void store_elem(void* base, size_t i, float x);
template <> __device__ __forceinline__ void store_elem<SAR_BF16>(void* base, size_t i, float x) {
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ void store_elem<SAR_FP16>(void* base, size_t i, float x) {
    static_cast<__half*>(base)[i] = __float2half_rn(x);
}
template <> __device__ __forceinline__ void store_elem<SAR_FP32>(void* base, size_t i, float x) {
    static_cast<float*>(base)[i] = x;
}
template <> __device__ __forceinline__ void store_elem<SAR_FP8_E4M3FN>(void* base, size_t i, float x) {
    static_cast<__nv_fp8_storage_t*>(base)[i] = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Widen element `e` of a 32-bit payload word (used by the LL tail).
template <int DT> __device__ __forceinline__ float widen_one(uint32_t w, int e) {
    float x[PerWord<DT>::kN];
    widen_word<DT>(w, x);
    return x[e];
}

// ---------------------------------------------------------------------------
// Global-memory access with streaming cache hints.  Every byte of the rsag
// inputs and outputs is touched exactly once, so nothing is kept in L1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// LL packets: two 8-byte packets per 16-byte access.  A vector access is two
// single-copy-atomic 8-byte accesses, so each packet's payload and flag are
// always observed together.  volatile keeps every poll a fresh read.
__device__ __forceinline__ void ld_packets2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint64_t ld_packet(const uint64_t* p) {
    uint64_t a;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void st_packets2(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" :: "l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_packet(uint64_t* p, uint64_t a) {
    asm volatile("st.volatile.global.u64 [%0], %1;" :: "l"(p), "l"(a) : "memory");
}

__device__ __forceinline__ uint64_t make_packet(uint32_t payload, uint32_t epoch) {
    return static_cast<uint64_t>(payload) | (static_cast<uint64_t>(epoch) << 32);
}
__device__ __forceinline__ uint32_t packet_flag(uint64_t p) { return static_cast<uint32_t>(p >> 32); }
__device__ __forceinline__ uint32_t packet_payload(uint64_t p) { return static_cast<uint32_t>(p); }

}  // namespace sar
