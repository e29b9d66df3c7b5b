/*
 * sar_oracle.c -- the CPU oracle for the simulated allreduce.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the package's smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares
 * no source, header, table or helper with the CUDA library; the two meet only
 * in the seeded input generator, which holds none of the arithmetic below.
 *
 * Plain, slow, single-threaded C11, built with -ffp-contract=off so that every
 * float operation below is exactly one IEEE binary32 operation with
 * round-to-nearest-even and gradual underflow.
 *
 * What it computes (and where that is stated):
 *
 *  - Allreduce.  "Support 2 ranks in AllreduceRsAgZeroCopy - #948", sections
 *    "why" and "what changed": ncclAllReduce semantics, i.e. every rank ends
 *    with the elementwise sum of all ranks' inputs; the rsag zero-copy kernel
 *    reduces a 1/N chunk per rank and writes it back to every peer.  Chunking
 *    never changes a value because every element is reduced on its own, so the
 *    oracle is the plain definition:
 *        out[j][i] = R_dt( (((f32(in[0][i]) + f32(in[1][i])) + ...) + f32(in[N-1][i])) )
 *    with the accumulator in binary32: mscclpp commit history, the summary
 *    "Add mixed-precision accumulation for allreduce" (accumDtype = float32 for
 *    low-precision inputs) and the ROCm FP8 summary ("higher-precision
 *    accumulation ... when reducing FP8 data").  f32() is exact widening and
 *    R_dt is one round-to-nearest-even into the element type.  The seed is
 *    acc = f32(in[0][i]) (not 0 + in[0][i]) so that nranks == 1 is the identity,
 *    -0 included; the rank order is 0..N-1 for every output.
 *
 *  - Reduce-scatter and all-gather steps of the rsag style (same page, "what
 *    changed"): rank r owns chunk r = [r*C, min(count, (r+1)*C)) where
 *    C = ceil(count / N) rounded up to a whole 16-byte vector of elements.
 *
 *  - LL packets.  mscclpp commit history, the allreduce_allpair_packet fix
 *    ("send/reduce/write-back" in one thread block, flag update logic): every
 *    4-byte payload travels with a 4-byte flag.  Packet w of rank r is 8 bytes:
 *    bytes 0..3 are bytes 4w..4w+3 of rank r's input (zero past the end of the
 *    input), bytes 4..7 the epoch as a little-endian uint32.  A packet whose
 *    flag differs from the epoch has not arrived; epoch 0 is reserved for a
 *    zeroed scratch that was never written (commit history, the TokenPool fix:
 *    recycled device counters must start from zero).
 *
 *  - Number formats, written from their definitions (not from any library):
 *      bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits; IEEE-style
 *                subnormals, infinities and NaNs.
 *      binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits (IEEE 754).
 *      e4m3fn  : OCP 8-bit floating point E4M3: 1 sign, 4 exponent (bias 7),
 *                3 fraction bits, no infinities, S.1111.111 is NaN, max finite
 *                S.1111.110 = 448, subnormals m/8 * 2^-6.  Conversion from
 *                binary32 saturates finite overflow and infinities to +-448
 *                ("satfinite"); NaN stays NaN.
 *      e4m3b15 : mscclpp commit history, "Add fp8_e4m3b15 datatype": 1 sign,
 *                4 exponent (bias 15), 3 fraction bits, max finite 0.9375.
 *                Max finite 0.9375 = 1.875 * 2^-1 puts the largest finite
 *                exponent field at 14, so field 15 is not finite; read
 *                IEEE-style: S.1111.000 = infinity, S.1111.mmm (mmm != 0) =
 *                NaN, subnormals m/8 * 2^-14, binary32 overflow rounds to
 *                infinity.
 *    Canonical NaN outputs: bf16 0x7FC0, fp16 0x7E00, e4m3fn 0x7F, e4m3b15
 *    0x7F, f32 0x7FC00000 (sign dropped).  Tests compare NaN by class.
 *
 * Parity pins (in the tests, independent of this file): brute-force nearest
 * search over each format's code table written from the field definitions,
 * library conversions, closed forms (N*x, nranks == 1 identity), exact
 * integer sums under rank permutation, exhaustive e4m3fn pairs, an
 * order-sensitive binary32 case, and the closed-form packet byte image.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element types; the integer codes are the oracle's own. */
enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP32 = 2, ORC_E4M3FN = 3, ORC_E4M3B15 = 4 };

/* Return codes. */
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_NOT_ARRIVED = 2 };

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

int orc_esize(int dt) {
    switch (dt) {
    case ORC_BF16: return 2;
    case ORC_FP16: return 2;
    case ORC_FP32: return 4;
    case ORC_E4M3FN: return 1;
    case ORC_E4M3B15: return 1;
    default: return 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Exact decoding: code -> binary32 value.                                   */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the top half of a binary32 with the same sign and exponent
 * fields, so the value of a code is the binary32 whose low 16 bits are zero. */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t e = (h >> 7) & 0xFF, f = h & 0x7F;
    if (e == 0xFF && f != 0) return bits_f32(0x7FC00000u);
    return bits_f32((uint32_t)h << 16);
}

/* binary16: E == 0 -> f * 2^-24; 0 < E < 31 -> (1024 + f) * 2^(E-25);
 * E == 31 -> infinity (f == 0) or NaN. */
float orc_fp16_to_f32(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    float mag;
    if (e == 0x1F) {
        if (f != 0) return bits_f32(0x7FC00000u);
        mag = INFINITY;
    } else if (e == 0) {
        mag = ldexpf((float)f, -24);
    } else {
        mag = ldexpf((float)(1024 + f), e - 25);
    }
    return s ? -mag : mag;
}

/* e4m3fn: E == 0 -> f * 2^-9; E > 0 -> (8 + f) * 2^(E-10); S.1111.111 -> NaN. */
float orc_e4m3fn_to_f32(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, f = c & 0x7;
    float mag;
    if (e == 0xF && f == 0x7) return bits_f32(0x7FC00000u);
    if (e == 0) mag = ldexpf((float)f, -9);
    else mag = ldexpf((float)(8 + f), e - 10);
    return s ? -mag : mag;
}

/* e4m3b15: E == 0 -> f * 2^-17; 0 < E < 15 -> (8 + f) * 2^(E-18);
 * E == 15 -> infinity (f == 0) or NaN. */
float orc_e4m3b15_to_f32(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, f = c & 0x7;
    float mag;
    if (e == 0xF) {
        if (f != 0) return bits_f32(0x7FC00000u);
        mag = INFINITY;
    } else if (e == 0) {
        mag = ldexpf((float)f, -17);
    } else {
        mag = ldexpf((float)(8 + f), e - 18);
    }
    return s ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* Rounding: binary32 -> narrower format, round to nearest, ties to even.    */
/* ------------------------------------------------------------------------ */

/*
 * A finite binary32 magnitude is sig * 2^exp with an integer significand
 * (24 bits for normals, the raw fraction for subnormals).  A target format
 * with p significand bits and minimum normal exponent emin has, in the binade
 * [2^e, 2^(e+1)), the quantum 2^(max(e, emin) - (p - 1)).  The rounded result
 * is n * 2^q with n = RNE(|x| / 2^q), an integer that fits p bits, or p+1 bits
 * when the rounding carried into the next binade (n == 2^p).
 */
typedef struct {
    int p;        /* significand bits including the implicit one */
    int emin;     /* exponent of the smallest normal */
    int bias;     /* exponent bias */
} orc_fmt;

/* Round |x| (finite, nonzero) to the format's grid: returns n and sets *q. */
static uint64_t round_to_grid(float ax, const orc_fmt* F, int* q_out) {
    uint32_t u = f32_bits(ax);
    uint32_t E = (u >> 23) & 0xFF, f = u & 0x7FFFFF;
    uint64_t sig;
    int exp2;                      /* value = sig * 2^exp2 */
    int e;                         /* floor(log2(value)) */
    if (E == 0) {                  /* binary32 subnormal */
        sig = f; exp2 = -149;
        e = -150; { uint64_t t = sig; while (t) { t >>= 1; e++; } }
    } else {
        sig = f | 0x800000u; exp2 = (int)E - 150;
        e = (int)E - 127;
    }
    int q = (e > F->emin ? e : F->emin) - (F->p - 1);
    int shift = q - exp2;          /* divide sig by 2^shift, round */
    uint64_t n;
    if (shift <= 0) {
        n = sig << (-shift);       /* exact, no rounding needed */
    } else if (shift > 40) {
        n = 0;                     /* below half a quantum: rounds to zero */
    } else {
        uint64_t keep = sig >> shift;
        uint64_t rest = sig & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        if (rest > half || (rest == half && (keep & 1))) keep += 1;
        n = keep;
    }
    *q_out = q;
    return n;
}

/* Assemble sign | exponent | fraction from n * 2^q; returns -1 on overflow of
 * the exponent field range [0, emax_field]. */
static int64_t encode_grid(uint64_t n, int q, const orc_fmt* F, int emax_field) {
    int fbits = F->p - 1;
    if (n == 0) return 0;
    if (n >= (1ull << F->p)) { n >>= 1; q += 1; }     /* carry into next binade */
    if (n < (1ull << fbits)) {                        /* subnormal: exponent field 0 */
        return (int64_t)n;
    }
    int field = q + fbits + F->bias;                  /* value = n * 2^q, n in [2^fbits, 2^p) */
    if (field > emax_field) return -1;
    return ((int64_t)field << fbits) | (int64_t)(n - (1ull << fbits));
}

uint16_t orc_f32_to_bf16(float x) {
    static const orc_fmt F = { 8, -126, 127 };
    uint32_t u = f32_bits(x);
    uint16_t s = (uint16_t)((u >> 16) & 0x8000);
    float ax = fabsf(x);
    if (isnan(x)) return 0x7FC0;
    if (isinf(x)) return s | 0x7F80;
    if (ax == 0.0f) return s;
    int q; uint64_t n = round_to_grid(ax, &F, &q);
    int64_t c = encode_grid(n, q, &F, 254);
    if (c < 0) return s | 0x7F80;                     /* overflow -> infinity */
    return s | (uint16_t)c;
}

uint16_t orc_f32_to_fp16(float x) {
    static const orc_fmt F = { 11, -14, 15 };
    uint32_t u = f32_bits(x);
    uint16_t s = (uint16_t)((u >> 16) & 0x8000);
    float ax = fabsf(x);
    if (isnan(x)) return 0x7E00;
    if (isinf(x)) return s | 0x7C00;
    if (ax == 0.0f) return s;
    int q; uint64_t n = round_to_grid(ax, &F, &q);
    int64_t c = encode_grid(n, q, &F, 30);
    if (c < 0) return s | 0x7C00;                     /* overflow -> infinity */
    return s | (uint16_t)c;
}

uint8_t orc_f32_to_e4m3fn(float x) {
    static const orc_fmt F = { 4, -6, 7 };
    uint32_t u = f32_bits(x);
    uint8_t s = (uint8_t)((u >> 24) & 0x80);
    float ax = fabsf(x);
    if (isnan(x)) return 0x7F;
    if (isinf(x)) return s | 0x7E;                    /* satfinite: +-448 */
    if (ax == 0.0f) return s;
    int q; uint64_t n = round_to_grid(ax, &F, &q);
    int64_t c = encode_grid(n, q, &F, 15);
    /* Exponent field 15 holds 256..448; fraction 111 there is NaN, so any
     * result above S.1111.110 saturates. */
    if (c < 0 || c > 0x7E) return s | 0x7E;
    return s | (uint8_t)c;
}

uint8_t orc_f32_to_e4m3b15(float x) {
    static const orc_fmt F = { 4, -14, 15 };
    uint32_t u = f32_bits(x);
    uint8_t s = (uint8_t)((u >> 24) & 0x80);
    float ax = fabsf(x);
    if (isnan(x)) return 0x7F;
    if (isinf(x)) return s | 0x78;
    if (ax == 0.0f) return s;
    int q; uint64_t n = round_to_grid(ax, &F, &q);
    int64_t c = encode_grid(n, q, &F, 14);
    if (c < 0) return s | 0x78;                       /* overflow -> infinity */
    return s | (uint8_t)c;
}

/* ------------------------------------------------------------------------ */
/* Element access on byte arrays.                                             */
/* ------------------------------------------------------------------------ */

float orc_load(int dt, const void* base, size_t i) {
    const uint8_t* b = (const uint8_t*)base;
    switch (dt) {
    case ORC_BF16: { uint16_t h; memcpy(&h, b + 2 * i, 2); return orc_bf16_to_f32(h); }
    case ORC_FP16: { uint16_t h; memcpy(&h, b + 2 * i, 2); return orc_fp16_to_f32(h); }
    case ORC_FP32: { float x; memcpy(&x, b + 4 * i, 4); return x; }
    case ORC_E4M3FN: return orc_e4m3fn_to_f32(b[i]);
    case ORC_E4M3B15: return orc_e4m3b15_to_f32(b[i]);
    }
    return NAN;
}

void orc_store(int dt, void* base, size_t i, float x) {
    uint8_t* b = (uint8_t*)base;
    switch (dt) {
    case ORC_BF16: { uint16_t h = orc_f32_to_bf16(x); memcpy(b + 2 * i, &h, 2); break; }
    case ORC_FP16: { uint16_t h = orc_f32_to_fp16(x); memcpy(b + 2 * i, &h, 2); break; }
    case ORC_FP32: {
        if (isnan(x)) x = bits_f32(0x7FC00000u);
        memcpy(b + 4 * i, &x, 4); break;
    }
    case ORC_E4M3FN: b[i] = orc_f32_to_e4m3fn(x); break;
    case ORC_E4M3B15: b[i] = orc_f32_to_e4m3b15(x); break;
    }
}

/* Bulk helpers for the tests. */
void orc_round_array(int dt, const float* x, void* y, size_t n) {
    for (size_t i = 0; i < n; ++i) orc_store(dt, y, i, x[i]);
}

void orc_decode_array(int dt, const void* x, float* y, size_t n) {
    for (size_t i = 0; i < n; ++i) y[i] = orc_load(dt, x, i);
}

/* Binary32 add as the oracle performs it (exposed so the tests can pin the
 * host's binary32 addition against exact rational sums). */
float orc_add_f32(float a, float b) { return a + b; }

/* ------------------------------------------------------------------------ */
/* The allreduce and its two rsag steps.                                     */
/* ------------------------------------------------------------------------ */

static int valid_args(int nranks, int dt) {
    return nranks >= 1 && nranks <= 32 && orc_esize(dt) != 0;
}

/* out[j][i] = R_dt(sum over k = 0..N-1 in order of f32(in[k][i])), all j. */
int orc_allreduce(const void* const* in, void* const* out, int nranks,
                  size_t count, int dt) {
    if (!valid_args(nranks, dt)) return ORC_BAD_ARG;
    for (size_t i = 0; i < count; ++i) {
        float acc = orc_load(dt, in[0], i);
        for (int k = 1; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);
        for (int j = 0; j < nranks; ++j) orc_store(dt, out[j], i, acc);
    }
    return ORC_OK;
}

/* Accumulation in another type (mscclpp commit history, "Add mixed-precision
 * accumulation for allreduce": accumDtype, with AUTO resolving to the input
 * type, and FP8 inputs reduced in float16 or float32).  Every partial sum is
 * rounded into the accumulator type:
 *     acc_0 = R_acc(f32(in[0][i]))
 *     acc_k = R_acc(f32(acc_{k-1}) + f32(in[k][i]))      (binary32 add, RNE)
 *     out[j][i] = R_dt(f32(acc_{N-1}))
 * acc_dt == ORC_FP32 is orc_allreduce; acc_dt == dt is native accumulation. */
static float round_through(int acc_dt, float x) {
    uint8_t tmp[4];
    orc_store(acc_dt, tmp, 0, x);
    return orc_load(acc_dt, tmp, 0);
}

int orc_allreduce_accum(const void* const* in, void* const* out, int nranks,
                        size_t count, int dt, int acc_dt) {
    if (!valid_args(nranks, dt) || orc_esize(acc_dt) == 0) return ORC_BAD_ARG;
    for (size_t i = 0; i < count; ++i) {
        float acc = round_through(acc_dt, orc_load(dt, in[0], i));
        for (int k = 1; k < nranks; ++k)
            acc = round_through(acc_dt, acc + orc_load(dt, in[k], i));
        for (int j = 0; j < nranks; ++j) orc_store(dt, out[j], i, acc);
    }
    return ORC_OK;
}

/* Chunk of simulated rank r: C = ceil(count / N) rounded up to a multiple of
 * the elements in 16 bytes; chunk r = [r*C, min(count, (r+1)*C)), possibly
 * empty. */
void orc_rsag_chunk(size_t count, int nranks, int dt, int r,
                    size_t* begin, size_t* end) {
    size_t vec = 16 / (size_t)orc_esize(dt);
    size_t c = (count + (size_t)nranks - 1) / (size_t)nranks;
    c = (c + vec - 1) / vec * vec;
    size_t b = (size_t)r * c, e = b + c;
    if (b > count) b = count;
    if (e > count) e = count;
    *begin = b; *end = e;
}

/* Reduce-scatter step: for every r, out[r][chunk r] = the reduced chunk.
 * Nothing else of any output is written. */
int orc_reduce_scatter(const void* const* in, void* const* out, int nranks,
                       size_t count, int dt) {
    if (!valid_args(nranks, dt)) return ORC_BAD_ARG;
    for (int r = 0; r < nranks; ++r) {
        size_t b, e;
        orc_rsag_chunk(count, nranks, dt, r, &b, &e);
        for (size_t i = b; i < e; ++i) {
            float acc = orc_load(dt, in[0], i);
            for (int k = 1; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);
            orc_store(dt, out[r], i, acc);
        }
    }
    return ORC_OK;
}

/* All-gather step: for every r and every j != r, out[j][chunk r] takes the
 * bytes of out[r][chunk r]. */
int orc_all_gather(void* const* out, int nranks, size_t count, int dt) {
    if (!valid_args(nranks, dt)) return ORC_BAD_ARG;
    size_t es = (size_t)orc_esize(dt);
    for (int r = 0; r < nranks; ++r) {
        size_t b, e;
        orc_rsag_chunk(count, nranks, dt, r, &b, &e);
        for (int j = 0; j < nranks; ++j) {
            if (j == r || e == b) continue;
            memmove((uint8_t*)out[j] + b * es, (const uint8_t*)out[r] + b * es,
                    (e - b) * es);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* LL packets.                                                               */
/* ------------------------------------------------------------------------ */

size_t orc_ll_packets(size_t count, int dt) {
    size_t bytes = count * (size_t)orc_esize(dt);
    return (bytes + 3) / 4;
}

/* Pack: packet w of rank r = {payload bytes 4w..4w+3 of in[r], epoch}. */
int orc_ll_pack(const void* const* in, void* const* pkts, int nranks,
                size_t count, int dt, uint32_t epoch) {
    if (!valid_args(nranks, dt) || epoch == 0) return ORC_BAD_ARG;
    size_t bytes = count * (size_t)orc_esize(dt);
    size_t np = orc_ll_packets(count, dt);
    for (int r = 0; r < nranks; ++r) {
        const uint8_t* src = (const uint8_t*)in[r];
        uint8_t* dst = (uint8_t*)pkts[r];
        for (size_t w = 0; w < np; ++w) {
            for (int k = 0; k < 4; ++k) {
                size_t at = 4 * w + (size_t)k;
                dst[8 * w + (size_t)k] = at < bytes ? src[at] : 0;
            }
            for (int k = 0; k < 4; ++k)
                dst[8 * w + 4 + (size_t)k] = (uint8_t)(epoch >> (8 * k));
        }
    }
    return ORC_OK;
}

/* Unpack-reduce: every packet of every rank must carry `epoch`; the payloads
 * rebuild each rank's input, which is then reduced exactly as orc_allreduce
 * does.  Returns ORC_NOT_ARRIVED (and writes nothing) if any flag differs. */
int orc_ll_unpack_reduce(const void* const* pkts, void* const* out, int nranks,
                         size_t count, int dt, uint32_t epoch) {
    if (!valid_args(nranks, dt) || epoch == 0) return ORC_BAD_ARG;
    size_t bytes = count * (size_t)orc_esize(dt);
    size_t np = orc_ll_packets(count, dt);
    for (int r = 0; r < nranks; ++r) {
        const uint8_t* p = (const uint8_t*)pkts[r];
        for (size_t w = 0; w < np; ++w) {
            uint32_t flag = (uint32_t)p[8 * w + 4] | ((uint32_t)p[8 * w + 5] << 8) |
                            ((uint32_t)p[8 * w + 6] << 16) | ((uint32_t)p[8 * w + 7] << 24);
            if (flag != epoch) return ORC_NOT_ARRIVED;
        }
    }
    uint8_t** rebuilt = (uint8_t**)calloc((size_t)nranks, sizeof(uint8_t*));
    if (!rebuilt) return ORC_BAD_ARG;
    int rc = ORC_OK;
    for (int r = 0; r < nranks; ++r) {
        rebuilt[r] = (uint8_t*)malloc(bytes ? bytes : 1);
        if (!rebuilt[r]) { rc = ORC_BAD_ARG; goto done; }
        const uint8_t* p = (const uint8_t*)pkts[r];
        for (size_t at = 0; at < bytes; ++at) rebuilt[r][at] = p[8 * (at / 4) + at % 4];
    }
    rc = orc_allreduce((const void* const*)rebuilt, out, nranks, count, dt);
done:
    for (int r = 0; r < nranks; ++r) free(rebuilt[r]);
    free(rebuilt);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Standalone conversion.                                                    */
/* ------------------------------------------------------------------------ */

/* dst[i] = R_dst(f32(src[i])): exact widening, one rounding. */
int orc_convert(const void* src, int src_dt, void* dst, int dst_dt, size_t count) {
    if (orc_esize(src_dt) == 0 || orc_esize(dst_dt) == 0) return ORC_BAD_ARG;
    for (size_t i = 0; i < count; ++i) orc_store(dst_dt, dst, i, orc_load(src_dt, src, i));
    return ORC_OK;
}
