// sar_device.cuh -- element types, 16-byte vector I/O and the in-order
// binary32 accumulation shared by the rsag and LL kernels.
//
// Arithmetic contract (mscclpp commit history, "Add mixed-precision
// accumulation for allreduce": FP8/16-bit inputs reduced in float32): every
// element is widened exactly to binary32, the ranks are added in order
// 0..N-1 with IEEE round-to-nearest-even adds (__fadd_rn: never contracted,
// never flushed; this library is built without fast-math or ftz), and the sum
// is rounded once to the element type: the hardware cvt.rn conversions for
// bf16, fp16 and e4m3fn (satfinite), software round-to-nearest-even for the
// e4m3b15 type, which has no hardware conversion (the rsag vector path instead
// runs e4m3b15 on the e4m3fn conversions, exactly, as described below).
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

// Kernels take the rank count as a template parameter NR, unrolled at compile
// time for 1, 2, 4, 8, 16 and 32 ranks; NR <= 0 marks a variant for any other
// count, passed at run time.
template <int NR> __device__ __forceinline__ int ranks(int n_rt) { return NR > 0 ? NR : n_rt; }

// Programmatic dependent launch (sm_90 and later).  The non-cooperative
// kernels are launched with programmatic stream serialization (launch_kernel
// in sar_internal.h), so a kernel can be scheduled while the one before it in
// the stream drains.  Each of them calls pdl_wait() before its first
// global-memory access: it returns once the preceding kernel has completed and
// its writes are visible, so stream order is kept exactly.  No kernel signals
// its dependents early (griddepcontrol.launch_dependents): measured, the early
// signal was no faster, and slower for the LL pair.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Element types.  kVE = elements per 16-byte vector.
// ---------------------------------------------------------------------------
template <int DT> struct Elem;
template <> struct Elem<SAR_BF16> { static constexpr int kSize = 2, kVE = 8; };
template <> struct Elem<SAR_FP16> { static constexpr int kSize = 2, kVE = 8; };
template <> struct Elem<SAR_FP32> { static constexpr int kSize = 4, kVE = 4; };
template <> struct Elem<SAR_FP8_E4M3FN> { static constexpr int kSize = 1, kVE = 16; };
template <> struct Elem<SAR_FP8_E4M3B15> { static constexpr int kSize = 1, kVE = 16; };

// e4m3b15 (1 sign, 4 exponent with bias 15, 3 fraction bits; exponent field
// 15 = infinity / NaN) has no hardware conversion; these follow the format's
// definition.  Widening places the 7 magnitude bits under the binary32
// exponent field, which reads them with bias 127, and rescales by 2^(127-15):
// exact for normals and subnormals alike.
__device__ __forceinline__ float e4m3b15_to_f32(uint32_t b) {
    const uint32_t em = b & 0x7Fu, sign = (b & 0x80u) << 24;
    const float finite = __uint_as_float(sign | (em << 20)) * 0x1p112f;
    const uint32_t special = em == 0x78u ? (sign | 0x7F800000u) : 0x7FFFFFFFu;   // inf or NaN
    return em >= 0x78u ? __uint_as_float(special) : finite;
}

// Narrowing: round to nearest even, overflow (|x| >= 0.96875, the midpoint
// above 0.9375) to infinity, NaN to 0x7F.  Branch-free: every candidate is
// computed and the right one selected.
__device__ __forceinline__ uint32_t f32_to_e4m3b15(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t sign = (u >> 24) & 0x80u, a = u & 0x7FFFFFFFu;
    // |x| < 2^-14: the subnormal grid of 2^-17 (exact scaling, then RNE).
    const uint32_t sub = __float2uint_rn(__uint_as_float(a) * 0x1p17f);
    // Normal: keep 3 fraction bits, ties to even; a carry moves into the
    // exponent.  Exponent fields differ by 127 - 15 = 112.
    const uint32_t r = a + 0x7FFFFu + ((a >> 20) & 1u);
    const uint32_t norm = (r >> 20) - (112u << 3);
    uint32_t m = a < 0x38800000u ? sub : norm;
    m = a >= 0x3F780000u ? 0x78u : m;                          // >= 0.96875: infinity
    return a > 0x7F800000u ? 0x7Fu : (sign | m);
}

// Exact widening of one 32-bit word holding 2 (16-bit types), 1 (fp32) or
// 4 (FP8 types) elements, lowest address first.
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

// Four codes one at a time (the rare words holding an infinity or NaN code);
// kept out of line so the unrolled reduction loops stay small.
static __device__ __noinline__ float4 e4m3b15_word_exact(uint32_t w) {
    return make_float4(e4m3b15_to_f32(w & 0xFFu), e4m3b15_to_f32((w >> 8) & 0xFFu),
                       e4m3b15_to_f32((w >> 16) & 0xFFu), e4m3b15_to_f32(w >> 24));
}

// e4m3b15 and binary16 share the bias 15, so a finite e4m3b15 code is the top
// of a binary16: sign to bit 15, exponent and fraction to bits 7..13.  Two
// codes become one f16x2 with a byte permute and two bit operations, then the
// hardware widens f16 -> f32 (exact).  Codes with exponent field 15 (infinity
// and NaN, which binary16 would read as 1.0 .. 1.875) take the per-code path;
// a SWAR test finds them: (code & 0x7F) + 8 carries into bit 7 exactly when
// the code's exponent field is 15.
template <> __device__ __forceinline__ void widen_word<SAR_FP8_E4M3B15>(uint32_t w, float* x) {
    if ((((w & 0x7F7F7F7Fu) + 0x08080808u) & 0x80808080u) == 0u) {
        const uint32_t b01 = __byte_perm(w, 0u, 0x1404), b23 = __byte_perm(w, 0u, 0x3424);   // [0,b0,0,b1], [0,b2,0,b3]
        uint32_t h01 = (b01 & 0x80008000u) | ((b01 & 0x7F007F00u) >> 1);
        uint32_t h23 = (b23 & 0x80008000u) | ((b23 & 0x7F007F00u) >> 1);
        const float2 f01 = __half22float2(*reinterpret_cast<__half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<__half2*>(&h23));
        x[0] = f01.x; x[1] = f01.y; x[2] = f23.x; x[3] = f23.y;
    } else {
        const float4 f = e4m3b15_word_exact(w);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    }
}
template <> __device__ __forceinline__ uint32_t narrow_word<SAR_FP8_E4M3B15>(const float* x) {
    return f32_to_e4m3b15(x[0]) | (f32_to_e4m3b15(x[1]) << 8) | (f32_to_e4m3b15(x[2]) << 16) |
           (f32_to_e4m3b15(x[3]) << 24);
}

// ---------------------------------------------------------------------------
// e4m3b15 on the e4m3fn hardware conversions (the vector path with a binary32
// accumulator).  The two formats have the same fields and differ in the bias
// (15 and 7) and in exponent field 15 (infinity and NaN in e4m3b15; 256..448
// and, with fraction 7, NaN in e4m3fn).  So a finite e4m3b15 code read as
// e4m3fn is its value times 2^8 exactly, subnormals included, and 2^8 times
// the e4m3b15 grid is the e4m3fn grid up to 240 = 2^8 * 0.9375.
//   * Sums.  Every e4m3b15 value is a multiple of 2^-17 of magnitude at most
//     0.9375, so a partial sum of up to 136 of them is a multiple of 2^-17
//     below 2^7 and exact in binary32 (24 bits), scaled or not:
//     the scaled sum is 2^8 times the sum, bit for bit, and infinities and
//     NaN combine the same way once the special codes are fixed up.
//   * Rounding.  Clamping 2^8 s to +-256 (NaN kept) and converting with the
//     saturating e4m3fn cvt rounds 2^8 s to the e4m3fn grid, which is 2^8
//     times rounding s to the e4m3b15 grid.  |s| >= 0.96875 (the overflow
//     threshold) lands on 256, whose code 0x78 is e4m3b15 infinity, and NaN
//     gives 0x7F.
// ---------------------------------------------------------------------------

static_assert(SAR_MAX_RANKS <= 136, "e4m3b15 sums on the e4m3fn path are exact only up to 136 ranks");

// True when any of the 16 codes has exponent field 15: (code & 0x7F) + 8
// carries into bit 7 exactly then, and never into the next byte.
__device__ __forceinline__ bool e4m3b15_vec_has_special(const uint4& v) {
    const uint32_t t = ((v.x & 0x7F7F7F7Fu) + 0x08080808u) | ((v.y & 0x7F7F7F7Fu) + 0x08080808u) |
                       ((v.z & 0x7F7F7F7Fu) + 0x08080808u) | ((v.w & 0x7F7F7F7Fu) + 0x08080808u);
    return (t & 0x80808080u) != 0u;
}

// 16 codes -> 2^8 times their values.  The e4m3fn reading of exponent field
// 15 is 256 (fraction 0: infinity here), 288..448 or NaN (fractions 1..7: NaN
// here); every other code reads at most 240.
__device__ __forceinline__ void e4m3b15_widen_scaled(const uint4& v, float* y) {
    widen_word<SAR_FP8_E4M3FN>(v.x, y + 0);
    widen_word<SAR_FP8_E4M3FN>(v.y, y + 4);
    widen_word<SAR_FP8_E4M3FN>(v.z, y + 8);
    widen_word<SAR_FP8_E4M3FN>(v.w, y + 12);
    if (e4m3b15_vec_has_special(v)) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float a = fabsf(y[e]);
            const float inf = copysignf(__int_as_float(0x7F800000), y[e]);
            y[e] = a == 256.0f ? inf : (a > 256.0f ? __int_as_float(0x7FFFFFFF) : y[e]);
        }
    }
}

// max(min(y, 256), -256), with NaN propagated (min.NaN / max.NaN).
__device__ __forceinline__ float clamp_256_keep_nan(float y) {
    const float hi = 256.0f, lo = -256.0f;
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(y), "f"(hi));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(r), "f"(lo));
    return r;
}

// 2^8 times binary32 sums -> one word of 4 e4m3b15 codes.
__device__ __forceinline__ uint32_t e4m3b15_narrow_scaled_word(const float* y) {
    const float c[4] = {clamp_256_keep_nan(y[0]), clamp_256_keep_nan(y[1]), clamp_256_keep_nan(y[2]),
                        clamp_256_keep_nan(y[3])};
    return narrow_word<SAR_FP8_E4M3FN>(c);
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

// The same three steps for e4m3b15 with the accumulator holding 2^8 times
// the binary32 sums (see e4m3b15_widen_scaled).
__device__ __forceinline__ void acc_seed_scaled(Acc<SAR_FP8_E4M3B15>& a, const uint4& v) {
    e4m3b15_widen_scaled(v, a.v);
}
__device__ __forceinline__ void acc_add_scaled(Acc<SAR_FP8_E4M3B15>& a, const uint4& v) {
    float y[16];
    e4m3b15_widen_scaled(v, y);
#pragma unroll
    for (int e = 0; e < 16; ++e) a.v[e] = __fadd_rn(a.v[e], y[e]);
}
__device__ __forceinline__ uint4 acc_round_scaled(const Acc<SAR_FP8_E4M3B15>& a) {
    return make_uint4(e4m3b15_narrow_scaled_word(a.v + 0), e4m3b15_narrow_scaled_word(a.v + 4),
                      e4m3b15_narrow_scaled_word(a.v + 8), e4m3b15_narrow_scaled_word(a.v + 12));
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

template <> __device__ __forceinline__ float load_elem<SAR_FP8_E4M3B15>(const void* base, size_t i) {
    return e4m3b15_to_f32(static_cast<const unsigned char*>(base)[i]);
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

template <> __device__ __forceinline__ void store_elem<SAR_FP8_E4M3B15>(void* base, size_t i, float x) {
    static_cast<unsigned char*>(base)[i] = static_cast<unsigned char>(f32_to_e4m3b15(x));
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

// L2 eviction priorities (createpolicy and the L2::cache_hint operand, sm_80
// and later).  The reduce-scatter step stores its chunk results as
// evict-last, so that the all-gather step that follows finds them in L2
// instead of reading them back from HBM; the all-gather reads them as
// evict-first, which hands those lines back to the normal eviction order.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_stream_hint(const uint4* p, uint64_t policy) {
    uint4 v;
    asm("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(policy));
    return v;
}
__device__ __forceinline__ void st_stream_hint(uint4* p, const uint4& v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

}  // namespace sar
