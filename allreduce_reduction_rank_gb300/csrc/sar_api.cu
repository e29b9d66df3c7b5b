// sar_api.cu -- the C ABI of libsar: argument validation, status codes and
// dispatch from the runtime rank count to the compile-time kernel variants.
//
// Every unsupported input is reported before anything is launched.  In
// "Support 2 ranks in AllreduceRsAgZeroCopy - #948" ("why") an unsupported
// rank count made the adapter return an error without launching, which the
// NCCL shim surfaced as ncclInvalidArgument; here the same condition is an
// explicit SAR_ERR_UNSUPPORTED_NRANKS.  The #948 set {2, 4, 8, 16, 32} (plus
// the trivial single rank) has compile-time-unrolled kernels; the counts that
// #948 still rejects (3, 5, 6, 7, ...) run kernels with a runtime rank loop.
#include <cstdint>
#include <cstring>

#include "sar_internal.h"

namespace sar {

size_t esize_of(sar_dtype dt) {
    switch (dt) {
    case SAR_BF16: return 2;
    case SAR_FP16: return 2;
    case SAR_FP32: return 4;
    case SAR_FP8_E4M3FN: return 1;
    case SAR_FP8_E4M3B15: return 1;
    }
    return 0;
}

namespace {

// Any count from 1 to SAR_MAX_RANKS: 1, 2, 4, 8, 16 and 32 run kernels with the
// rank loops unrolled at compile time, every other count a kernel that loops
// over the ranks at run time (same order, same results).
bool supported_nranks(int n) { return n >= 1 && n <= SAR_MAX_RANKS; }

bool valid_dtype(int dt) { return dt >= SAR_BF16 && dt <= SAR_FP8_E4M3B15; }

bool is_fp8(int dt) { return dt == SAR_FP8_E4M3FN || dt == SAR_FP8_E4M3B15; }

// Poll bound of sar_allreduce with SAR_ALGO_LL_ALLPAIR (re-reads of one packet,
// with sleeps of up to about a microsecond between them).  Every packet a poll
// waits for is sent by the same CTA, so the bound is never reached.
constexpr uint64_t kAllpairSpins = uint64_t(1) << 20;

// SAR_ALGO_LL_ALLPAIR runs the sliced shared-memory kernel, except for rank
// counts without an unrolled kernel (3, 5, 6, 7, 9, ...) from 4 ranks up to
// kCtaAllpairBytes over all ranks (N x S), which run in one CTA.  Measured
// (CUDA graph, us per call, one CTA / sliced): 8 x 1 KiB fp32 1.56 / 1.26,
// 4 x 2 KiB 1.56 / 1.13, 5 x 1 KiB 1.78 / 1.87, 6 x 1 KiB 1.86 / 1.98,
// 7 x 1 KiB 1.87 / 2.04.
constexpr size_t kCtaAllpairBytes = size_t(8) << 10;

bool unrolled_nranks(int n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks nranks device pointers: non-NULL and aligned to `align`; clears
// *all16 if any pointer is not 16-byte aligned.
sar_status check_ptrs(const void* const* arr, int nranks, size_t align, bool* all16) {
    for (int r = 0; r < nranks; ++r) {
        if (arr[r] == nullptr) return SAR_ERR_INVALID_ARG;
        if (!aligned(arr[r], align)) return SAR_ERR_MISALIGNED;
        if (!aligned(arr[r], 16)) *all16 = false;
    }
    return SAR_OK;
}

// Largest count for which the byte sizes (x8 for packet buffers) fit size_t.
bool count_fits(size_t count, size_t esize) { return count <= (SIZE_MAX / 16) / esize; }

sar_status to_status(cudaError_t e) { return e == cudaSuccess ? SAR_OK : SAR_ERR_CUDA; }

size_t rsag_chunk(size_t count, int nranks, sar_dtype dt) {
    const size_t vec = 16 / esize_of(dt);
    size_t c = (count + static_cast<size_t>(nranks) - 1) / static_cast<size_t>(nranks);
    return (c + vec - 1) / vec * vec;
}

// Common checks of the rsag entry points.  On SAR_OK with *launch == false
// there is nothing to do (count == 0).
sar_status check_rsag(const void* const* in, void* const* out, int nranks, size_t count, int dtype,
                      bool need_in, RankPtrs* p, bool* vec, bool* launch) {
    *launch = false;
    if (!supported_nranks(nranks)) return SAR_ERR_UNSUPPORTED_NRANKS;
    if (!valid_dtype(dtype)) return SAR_ERR_UNSUPPORTED_DTYPE;
    if ((need_in && in == nullptr) || out == nullptr) return SAR_ERR_INVALID_ARG;
    const size_t es = esize_of(static_cast<sar_dtype>(dtype));
    if (!count_fits(count, es)) return SAR_ERR_INVALID_ARG;
    if (count == 0) return SAR_OK;
    bool all16 = true;
    sar_status st;
    if (need_in && (st = check_ptrs(in, nranks, es, &all16)) != SAR_OK) return st;
    if ((st = check_ptrs(out, nranks, es,
                         &all16)) != SAR_OK)
        return st;
    std::memset(p, 0, sizeof(*p));
    for (int r = 0; r < nranks; ++r) {
        if (need_in) p->in[r] = in[r];
        p->out[r] = out[r];
    }
    *vec = all16;
    *launch = true;
    return SAR_OK;
}

// Buffers that are not all 16-byte aligned but share one misalignment (every
// address equal mod 16, as for slices at the same element offset of aligned
// buffers): the first `head` elements, up to the 16-byte boundary, go to the
// element kernels and the rest to the vector kernels on pointers advanced by
// `head`.  Every element is reduced on its own, so the values are those of one
// pass; the split only decides which kernel runs.  Returns 0 when it does not
// apply.
size_t common_head(const RankPtrs& p, int nranks, size_t count, size_t es) {
    const uintptr_t m = reinterpret_cast<uintptr_t>(p.out[0]) & 15u;
    if (m == 0 || m % es != 0) return 0;
    for (int r = 0; r < nranks; ++r)
        if ((reinterpret_cast<uintptr_t>(p.in[r]) & 15u) != m || (reinterpret_cast<uintptr_t>(p.out[r]) & 15u) != m)
            return 0;
    const size_t head = (16 - m) / es;
    return head < count ? head : 0;
}

RankPtrs advance(const RankPtrs& p, int nranks, size_t bytes) {
    RankPtrs q;
    std::memset(&q, 0, sizeof(q));
    for (int r = 0; r < nranks; ++r) {
        q.in[r] = static_cast<const char*>(p.in[r]) + bytes;
        q.out[r] = static_cast<char*>(p.out[r]) + bytes;
    }
    return q;
}

// Runs `launch(p, count, vec)` once, or twice (element-wise head, then the
// vectors) when the buffers share a misalignment.
template <class F>
sar_status split_by_alignment(const RankPtrs& p, int nranks, size_t count, size_t es, bool vec, F&& launch) {
    const size_t head = vec ? 0 : common_head(p, nranks, count, es);
    if (head == 0) return launch(p, count, vec);
    const sar_status st = launch(p, head, false);
    if (st != SAR_OK) return st;
    return launch(advance(p, nranks, head * es), count - head, true);
}

// Common checks of the LL entry points: rank count, element type, epoch,
// packet buffers (16-byte aligned) and the buffers of one side (`data`: the
// inputs of pack, the outputs of unpack-reduce).  *data16 tells whether every
// data buffer is 16-byte aligned.  On SAR_OK with *launch == false there is
// nothing to do (count == 0).
sar_status check_ll(const void* const* data, const void* const* pkts, int nranks, size_t count, int dtype,
                    uint32_t epoch, bool* launch, bool* data16) {
    *launch = false;
    if (!supported_nranks(nranks)) return SAR_ERR_UNSUPPORTED_NRANKS;
    if (!valid_dtype(dtype)) return SAR_ERR_UNSUPPORTED_DTYPE;
    if (data == nullptr || pkts == nullptr || epoch == 0) return SAR_ERR_INVALID_ARG;
    const size_t es = esize_of(static_cast<sar_dtype>(dtype));
    if (!count_fits(count, es)) return SAR_ERR_INVALID_ARG;
    if (count == 0) return SAR_OK;
    bool all16 = true, pk16 = true;
    sar_status st;
    if ((st = check_ptrs(data, nranks, es, &all16)) != SAR_OK) return st;
    if ((st = check_ptrs(pkts, nranks, 16, &pk16)) != SAR_OK) return st;
    *data16 = all16;
    *launch = true;
    return SAR_OK;
}

sar_status check_status_args(uint64_t max_spins, const int32_t* d_status) {
    if (d_status == nullptr || max_spins == 0) return SAR_ERR_INVALID_ARG;
    if (!aligned(d_status, 4)) return SAR_ERR_MISALIGNED;
    return SAR_OK;
}

// The LL allreduce (pack, then poll/unpack/reduce) on the packet scratch
// `pkts`; with `two_halves` the scratch is double-buffered and the call uses
// half (epoch & 1), each half being the packet bytes rounded up to 16.
sar_status allreduce_ll(const void* const* in, void* const* out, void* const* pkts, int nranks, size_t count,
                        sar_dtype dtype, uint32_t epoch, uint64_t max_spins, int32_t* d_status, sar_stream_t stream,
                        bool two_halves) {
    bool launch = false, in16 = false, out16 = false;
    sar_status st = check_ll(in, pkts, nranks, count, dtype, epoch, &launch, &in16);
    if (st != SAR_OK) return st;
    if (out == nullptr) return SAR_ERR_INVALID_ARG;
    if ((st = check_status_args(max_spins, d_status)) != SAR_OK) return st;
    if (!launch) return SAR_OK;
    if ((st = check_ll(out, pkts, nranks, count, dtype, epoch, &launch, &out16)) != SAR_OK) return st;
    const size_t half = ((count * esize_of(dtype) + 3) / 4 * 8 + 15) / 16 * 16;
    const size_t offset = two_halves ? (epoch & 1u) * half : 0;
    RankPtrs pack, unpack;
    std::memset(&pack, 0, sizeof(pack));
    std::memset(&unpack, 0, sizeof(unpack));
    for (int r = 0; r < nranks; ++r) {
        void* pk = static_cast<char*>(pkts[r]) + offset;
        pack.in[r] = in[r];
        pack.out[r] = pk;
        unpack.in[r] = pk;
        unpack.out[r] = out[r];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = to_status(launch_ll_pack(nranks, pack, count * esize_of(dtype), epoch, in16, s));
    if (st != SAR_OK) return st;
    return to_status(
        launch_ll_unpack_reduce(dtype, nranks, unpack, count, epoch, max_spins, d_status, out16, s));
}

}  // namespace
}  // namespace sar

using namespace sar;

extern "C" {

SAR_API size_t sar_rsag_chunk(size_t count, int nranks, sar_dtype dtype) {
    if (!supported_nranks(nranks) || !valid_dtype(dtype)) return 0;
    return rsag_chunk(count, nranks, dtype);
}

SAR_API sar_status sar_allreduce(const void* const* in, void* const* out, int nranks, size_t count,
                                 sar_dtype dtype, sar_algo algo, sar_stream_t stream) {
    if (algo == SAR_ALGO_LL_ALLPAIR) {
        // One launch, every packet in the shared memory of the CTA that made
        // and polls it: no scratch and no state, so calls may overlap and be
        // captured anywhere.
        RankPtrs p;
        bool vec = false, launch = false;
        const sar_status st = check_rsag(in, out, nranks, count, dtype, true, &p, &vec, &launch);
        if (st != SAR_OK || !launch) return st;
        bool in16 = true, out16 = true;
        for (int r = 0; r < nranks; ++r) {
            in16 = in16 && aligned(in[r], 16);
            out16 = out16 && aligned(out[r], 16);
        }
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (!unrolled_nranks(nranks) && nranks >= 4 &&
            count * esize_of(dtype) <= kCtaAllpairBytes / static_cast<size_t>(nranks) &&
            ll_cta_slot_bytes(nranks, count, dtype) <= kLLCtaMaxSlotBytes)
            return to_status(launch_ll_cta(dtype, nranks, p, count, kAllpairSpins, nullptr, in16, out16, s));
        return to_status(launch_ll_slice(dtype, nranks, p, count, kAllpairSpins, nullptr, in16, out16, s));
    }
    if (algo != SAR_ALGO_RSAG && algo != SAR_ALGO_RSAG_TWO_PHASE) {
        if (!supported_nranks(nranks)) return SAR_ERR_UNSUPPORTED_NRANKS;
        return SAR_ERR_INVALID_ARG;
    }
    RankPtrs p;
    bool vec = false, launch = false;
    sar_status st = check_rsag(in, out, nranks, count, dtype, true, &p, &vec, &launch);
    if (st != SAR_OK || !launch) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return split_by_alignment(p, nranks, count, esize_of(dtype), vec, [&](const RankPtrs& q, size_t n, bool v) {
        const size_t chunk = rsag_chunk(n, nranks, dtype);
        if (algo == SAR_ALGO_RSAG) return to_status(launch_rsag(kFused, dtype, nranks, q, n, chunk, v, s));
        const sar_status r = to_status(launch_rsag(kReduceScatter, dtype, nranks, q, n, chunk, v, s));
        if (r != SAR_OK) return r;
        return to_status(launch_all_gather(nranks, q, n, esize_of(dtype), chunk, v, s));
    });
}

SAR_API sar_status sar_allreduce_accum(const void* const* in, void* const* out, int nranks, size_t count,
                                       sar_dtype dtype, sar_dtype accum, sar_stream_t stream) {
    if (!valid_dtype(accum)) return SAR_ERR_UNSUPPORTED_DTYPE;
    const bool narrow = accum == SAR_FP16 || accum == SAR_BF16 || (accum == dtype);
    if (accum != SAR_FP32 && !narrow) return SAR_ERR_UNSUPPORTED_DTYPE;
    RankPtrs p;
    bool vec = false, launch = false;
    sar_status st = check_rsag(in, out, nranks, count, dtype, true, &p, &vec, &launch);
    if (st != SAR_OK || !launch) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return split_by_alignment(p, nranks, count, esize_of(dtype), vec, [&](const RankPtrs& q, size_t n, bool v) {
        const size_t chunk = rsag_chunk(n, nranks, dtype);
        if (accum == SAR_FP32) return to_status(launch_rsag(kFused, dtype, nranks, q, n, chunk, v, s));
        return to_status(launch_rsag_accum(dtype, accum, nranks, q, n, chunk, v, s));
    });
}

SAR_API sar_status sar_reduce_scatter(const void* const* in, void* const* out, int nranks, size_t count,
                                      sar_dtype dtype, sar_stream_t stream) {
    RankPtrs p;
    bool vec = false, launch = false;
    sar_status st = check_rsag(in, out, nranks, count, dtype, true, &p, &vec, &launch);
    if (st != SAR_OK || !launch) return st;
    return to_status(launch_rsag(kReduceScatter, dtype, nranks, p, count, rsag_chunk(count, nranks, dtype), vec,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_all_gather(void* const* out, int nranks, size_t count, sar_dtype dtype,
                                  sar_stream_t stream) {
    RankPtrs p;
    bool vec = false, launch = false;
    sar_status st = check_rsag(nullptr, out, nranks, count, dtype, false, &p, &vec, &launch);
    if (st != SAR_OK || !launch) return st;
    return to_status(launch_all_gather(nranks, p, count, esize_of(dtype), rsag_chunk(count, nranks, dtype), vec,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API size_t sar_ll_packet_bytes(size_t count, sar_dtype dtype) {
    if (!valid_dtype(dtype)) return 0;
    const size_t es = esize_of(dtype);
    if (!count_fits(count, es)) return 0;
    return (count * es + 3) / 4 * 8;
}

SAR_API sar_status sar_ll_pack(const void* const* in, void* const* pkts, int nranks, size_t count,
                               sar_dtype dtype, uint32_t epoch, sar_stream_t stream) {
    bool launch = false, in16 = false;
    sar_status st = check_ll(in, pkts, nranks, count, dtype, epoch, &launch, &in16);
    if (st != SAR_OK || !launch) return st;
    RankPtrs p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = in[r];
        p.out[r] = pkts[r];
    }
    return to_status(launch_ll_pack(nranks, p, count * esize_of(dtype), epoch, in16,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_ll_unpack_reduce(const void* const* pkts, void* const* out, int nranks, size_t count,
                                        sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                                        int32_t* d_status, sar_stream_t stream) {
    bool launch = false, out16 = false;
    sar_status st = check_ll(out, pkts, nranks, count, dtype, epoch, &launch, &out16);
    if (st != SAR_OK) return st;
    if ((st = check_status_args(max_spins, d_status)) != SAR_OK) return st;
    if (!launch) return SAR_OK;
    RankPtrs p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = pkts[r];
        p.out[r] = out[r];
    }
    return to_status(launch_ll_unpack_reduce(dtype, nranks, p, count, epoch, max_spins, d_status, out16,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_allreduce_ll(const void* const* in, void* const* out, void* const* pkts, int nranks,
                                    size_t count, sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                                    int32_t* d_status, sar_stream_t stream) {
    return allreduce_ll(in, out, pkts, nranks, count, dtype, epoch, max_spins, d_status, stream, false);
}

SAR_API sar_status sar_allreduce_ll_double(const void* const* in, void* const* out, void* const* pkts, int nranks,
                                           size_t count, sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                                           int32_t* d_status, sar_stream_t stream) {
    return allreduce_ll(in, out, pkts, nranks, count, dtype, epoch, max_spins, d_status, stream, true);
}

SAR_API sar_status sar_allreduce_ll_fused(const void* const* in, void* const* out, void* const* pkts, int nranks,
                                          size_t count, sar_dtype dtype, uint32_t epoch, uint64_t* d_epoch,
                                          uint64_t max_spins, int32_t* d_status, sar_stream_t stream) {
    bool launch = false, in16 = false, out16 = false;
    // With a device epoch counter the host epoch is unused; any non-zero value
    // passes the shared check.
    sar_status st = check_ll(in, pkts, nranks, count, dtype, d_epoch != nullptr ? 1u : epoch, &launch, &in16);
    if (st != SAR_OK) return st;
    if (out == nullptr) return SAR_ERR_INVALID_ARG;
    if ((st = check_status_args(max_spins, d_status)) != SAR_OK) return st;
    if (d_epoch != nullptr && !aligned(d_epoch, 8)) return SAR_ERR_MISALIGNED;
    if (!launch) return SAR_OK;
    if ((st = check_ll(out, pkts, nranks, count, dtype, 1u, &launch, &out16)) != SAR_OK) return st;
    RankPtrs data;
    std::memset(&data, 0, sizeof(data));
    for (int r = 0; r < nranks; ++r) {
        data.in[r] = in[r];
        data.out[r] = out[r];
    }
    return to_status(launch_ll_fused(dtype, nranks, data, pkts, count, epoch, d_epoch, max_spins, d_status, in16,
                                     out16, reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_allreduce_ll_writeback(const void* const* in, void* const* out, void* const* pkts, void* res,
                                              int nranks, size_t count, sar_dtype dtype, uint32_t epoch,
                                              uint64_t* d_epoch, int multi_dest, uint64_t max_spins,
                                              int32_t* d_status, sar_stream_t stream) {
    bool launch = false, in16 = false, out16 = false;
    sar_status st = check_ll(in, pkts, nranks, count, dtype, d_epoch != nullptr ? 1u : epoch, &launch, &in16);
    if (st != SAR_OK) return st;
    if (out == nullptr) return SAR_ERR_INVALID_ARG;
    if ((st = check_status_args(max_spins, d_status)) != SAR_OK) return st;
    if (d_epoch != nullptr && !aligned(d_epoch, 8)) return SAR_ERR_MISALIGNED;
    if (!launch) return SAR_OK;
    if (res == nullptr) return SAR_ERR_INVALID_ARG;
    if (!aligned(res, 16)) return SAR_ERR_MISALIGNED;
    if ((st = check_ll(out, pkts, nranks, count, dtype, 1u, &launch, &out16)) != SAR_OK) return st;
    RankPtrs data;
    std::memset(&data, 0, sizeof(data));
    for (int r = 0; r < nranks; ++r) {
        data.in[r] = in[r];
        data.out[r] = out[r];
    }
    return to_status(launch_ll_writeback(dtype, nranks, data, pkts, res, count, epoch, d_epoch, multi_dest != 0,
                                         max_spins, d_status, in16, out16, reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_allreduce_ll_cluster(const void* const* in, void* const* out, int nranks, size_t count,
                                            sar_dtype dtype, uint64_t max_spins, int32_t* d_status,
                                            sar_stream_t stream) {
    if (nranks < 1 || nranks > SAR_LL_CLUSTER_MAX_RANKS) return SAR_ERR_UNSUPPORTED_NRANKS;
    RankPtrs p;
    bool vec = false, launch = false;
    sar_status st = check_rsag(in, out, nranks, count, dtype, true, &p, &vec, &launch);
    if (st != SAR_OK) return st;
    if ((st = check_status_args(max_spins, d_status)) != SAR_OK) return st;
    if (!launch) return SAR_OK;
    bool in16 = true, out16 = true;
    for (int r = 0; r < nranks; ++r) {
        in16 = in16 && aligned(in[r], 16);
        out16 = out16 && aligned(out[r], 16);
    }
    return to_status(launch_ll_cluster(dtype, nranks, p, count, max_spins, d_status, in16, out16,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_fp8_convert(const void* src, sar_dtype src_dtype, void* dst, sar_dtype dst_dtype,
                                   size_t count, sar_stream_t stream) {
    if (!valid_dtype(src_dtype) || !valid_dtype(dst_dtype)) return SAR_ERR_UNSUPPORTED_DTYPE;
    // One side FP8, the other fp32, fp16 or bf16.
    const bool pair_ok = is_fp8(src_dtype) != is_fp8(dst_dtype);
    if (!pair_ok) return SAR_ERR_UNSUPPORTED_DTYPE;
    if (src == nullptr || dst == nullptr) return SAR_ERR_INVALID_ARG;
    const size_t ses = esize_of(src_dtype), des = esize_of(dst_dtype);
    if (!count_fits(count, 4)) return SAR_ERR_INVALID_ARG;
    if (!aligned(src, ses) || !aligned(dst, des)) return SAR_ERR_MISALIGNED;
    if (count == 0) return SAR_OK;
    const bool vec = aligned(src, 16) && aligned(dst, 16);
    return to_status(launch_convert(src, src_dtype, dst, dst_dtype, count, vec,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

SAR_API sar_status sar_read_device_status(const int32_t* d_status, sar_stream_t stream) {
    if (d_status == nullptr) return SAR_ERR_INVALID_ARG;
    int32_t h = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, d_status, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SAR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SAR_ERR_CUDA;
    if (h == 0) return SAR_OK;
    if (h == SAR_ERR_TIMEOUT) return SAR_ERR_TIMEOUT;
    return SAR_ERR_CUDA;
}

SAR_API const char* sar_status_string(sar_status status) {
    switch (status) {
    case SAR_OK: return "SAR_OK";
    case SAR_ERR_INVALID_ARG: return "SAR_ERR_INVALID_ARG: invalid argument";
    case SAR_ERR_UNSUPPORTED_NRANKS: return "SAR_ERR_UNSUPPORTED_NRANKS: nranks must be between 1 and 32";
    case SAR_ERR_UNSUPPORTED_DTYPE: return "SAR_ERR_UNSUPPORTED_DTYPE: unsupported element type or conversion";
    case SAR_ERR_MISALIGNED: return "SAR_ERR_MISALIGNED: buffer not aligned to its element (packets: 16 bytes)";
    case SAR_ERR_CUDA: return "SAR_ERR_CUDA: a CUDA launch or copy failed";
    case SAR_ERR_TIMEOUT: return "SAR_ERR_TIMEOUT: an LL flag poll ran out of spins";
    }
    return "unknown sar_status";
}

}  // extern "C"
