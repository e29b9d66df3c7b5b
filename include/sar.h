/*
 * sar.h -- libsar, the simulated allreduce on one GB300 (sm_103a).
 *
 * N simulated ranks are N separate buffers in the HBM of one GPU.  The library
 * computes the data-parallel hot path of the MSCCL++ allreduce algorithms: the
 * N-way elementwise sum of the ranks' buffers, accumulated in binary32 and
 * rounded once to the element type, in two styles:
 *
 *   rsag  - reduce-scatter then all-gather ("Support 2 ranks in
 *           AllreduceRsAgZeroCopy - #948", sections "why" and "what changed":
 *           each rank reduces its 1/N chunk of every peer's input and writes
 *           the result back to every peer's output);
 *   LL    - all-pair low-latency packets (mscclpp commit history, the
 *           allreduce_allpair_packet fix: send, reduce and write-back in one
 *           thread block, with flag-checked packets).
 *
 * Accumulation is binary32 (mscclpp commit history, "Add mixed-precision
 * accumulation for allreduce": accumDtype), summed in rank order 0..N-1 for
 * every element and every output, then rounded once with round-to-nearest-
 * even; sar_allreduce_accum instead rounds every partial sum into a narrower
 * accumulator.  Results are therefore reproducible bit for bit.
 *
 * Conventions shared by every entry point:
 *  - Pointer arrays (`in`, `out`, `pkts`) are HOST arrays of `nranks` DEVICE
 *    pointers.  The caller owns the arrays and every buffer.  The library
 *    copies the pointers into kernel parameters, keeps no caller pointer after
 *    the call returns, allocates nothing and does not synchronise (except
 *    sar_read_device_status), so calls are stream-ordered and may be captured
 *    into a CUDA graph.  The only state kept between calls belongs to
 *    sar_allreduce_ll_noalloc: the fixed packet scratch compiled into the
 *    library and, per device, its address and last epoch.
 *  - `count` is the number of elements per rank.  count == 0 returns SAR_OK
 *    without launching anything.
 *  - Every argument error is returned before any launch.  nranks may be any
 *    count from 1 to SAR_MAX_RANKS (32); other values return
 *    SAR_ERR_UNSUPPORTED_NRANKS and launch nothing.  1, 2, 4, 8, 16 and 32
 *    ranks run kernels with the rank loops unrolled at compile time (in #948
 *    the rsag kernel exists only for 2, 4, 8, 16 and 32 ranks and other counts
 *    returned an error without launching); every other count runs a kernel
 *    that loops over the ranks at run time, in the same order, with the same
 *    results.
 *  - Buffers must be aligned to their element size (else SAR_ERR_MISALIGNED).
 *    When every buffer of a call is 16-byte aligned the kernels move 16-byte
 *    vectors.  sar_allreduce and sar_allreduce_accum also do when every buffer
 *    has the same address modulo 16 (the elements up to the 16-byte boundary
 *    run element-wise); otherwise a slower element-wise kernel runs.  Results
 *    are identical either way.
 *  - A failed launch returns SAR_ERR_CUDA.
 *  - Kernels are launched with programmatic stream serialization (programmatic
 *    dependent launch): one may be scheduled while the work before it in the
 *    stream drains, but it waits for that work to complete (griddepcontrol.
 *    wait) before touching memory, so stream order and results are exactly
 *    those of plain launches.  No library kernel signals its dependents early.
 *  - `stream` is a CUDA stream (cudaStream_t); NULL is the legacy default
 *    stream.  The current device must be the one that owns the buffers.
 */
#ifndef SAR_H_
#define SAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SAR_API __attribute__((visibility("default")))
#else
#define SAR_API
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* sar_stream_t;

#define SAR_MAX_RANKS 32

typedef enum {
    SAR_BF16 = 0,        /* bfloat16, 2 bytes */
    SAR_FP16 = 1,        /* IEEE binary16, 2 bytes */
    SAR_FP32 = 2,        /* IEEE binary32, 4 bytes */
    SAR_FP8_E4M3FN = 3,  /* OCP FP8 E4M3 (bias 7, no inf, NaN = S.1111.111,
                            max +-448; binary32 -> e4m3fn saturates), 1 byte */
    SAR_FP8_E4M3B15 = 4  /* software FP8, bias 15, max finite 0.9375 (mscclpp
                            commit history, "Add fp8_e4m3b15 datatype");
                            S.1111.000 = inf, S.1111.mmm = NaN, binary32
                            overflow rounds to inf, subnormals m/8 * 2^-14 */
} sar_dtype;

typedef enum {
    SAR_ALGO_RSAG = 0,            /* one fused kernel: reduce chunk, write to all outputs */
    SAR_ALGO_RSAG_TWO_PHASE = 1,  /* reduce-scatter kernel, then all-gather kernel */
    SAR_ALGO_LL_ALLPAIR = 2       /* LL all-pair packets in shared memory, one launch */
} sar_algo;

typedef enum {
    SAR_OK = 0,
    SAR_ERR_INVALID_ARG = 1,        /* NULL pointer, bad enum, epoch 0, size overflow, ... */
    SAR_ERR_UNSUPPORTED_NRANKS = 2, /* nranks outside 1..SAR_MAX_RANKS */
    SAR_ERR_UNSUPPORTED_DTYPE = 3,  /* dtype (or conversion pair) not supported */
    SAR_ERR_MISALIGNED = 4,         /* buffer not aligned to its element size (16 B for packets) */
    SAR_ERR_CUDA = 5,               /* a CUDA launch or copy failed */
    SAR_ERR_TIMEOUT = 6             /* an LL flag poll ran out of spins (reported on the device) */
} sar_status;

/*
 * sar_allreduce -- the allreduce, by the rsag algorithm (fused or two-phase)
 * or the LL all-pair algorithm.
 *
 * rsag is defined by "Support 2 ranks in AllreduceRsAgZeroCopy - #948"
 * ("why": the ncclAllReduce that the rsag zero-copy algorithm serves; "what
 * changed": NPeers = NRanks - 1, peer loops unrolled at compile time).
 *
 * For every element i and every rank j:
 *   out[j][i] = R( (((f32(in[0][i]) + f32(in[1][i])) + f32(in[2][i])) ... + f32(in[N-1][i])) )
 * with binary32 additions and one round-to-nearest-even R into `dtype`
 * (e4m3fn saturates to +-448).
 *
 * Simulated rank r owns chunk r = [r*C, min(count, (r+1)*C)) where
 * C = sar_rsag_chunk(count, nranks, dtype).  SAR_ALGO_RSAG reduces each chunk
 * and writes it to all N outputs in one kernel (N*S bytes read, N*S written,
 * S = count * element size).  SAR_ALGO_RSAG_TWO_PHASE runs sar_reduce_scatter
 * then sar_all_gather.
 *
 * SAR_ALGO_LL_ALLPAIR runs the LL all-pair allreduce (mscclpp commit history,
 * the allreduce_allpair_packet fix: send, reduce and write-back in the same
 * thread block, packets checked by their flags) in one launch, with every
 * packet in the shared memory of the CTA that makes and polls it:
 *  - by default, CTA b plays every rank for one slice of the packets: it turns
 *    the slice of each rank's input into {payload, flag} packets in its
 *    shared memory, polls each packet's flag, reduces in rank order and writes
 *    the result to all N outputs, so a call of any size spreads over the SMs;
 *  - for rank counts without an unrolled kernel (3, 5, 6, 7, 9, ...) from 4
 *    ranks up to 8 KiB over all ranks (nranks * S), one CTA plays every rank
 *    for the whole call (measured faster there).
 * Neither form uses scratch or keeps state: calls may overlap on the GPU and
 * may be captured into a CUDA graph at any time.  Every packet a poll waits
 * for is sent by the same CTA, so the polls' bound is never reached in a
 * correct call.  Any size whose buffers exist is accepted.
 *
 * All three algorithms give the same bits.
 *
 * in, out : host arrays of `nranks` device pointers, `count` elements each,
 *           dense.  out[r] == in[r] (in place) is allowed; any other overlap
 *           between buffers is undefined.
 */
SAR_API sar_status sar_allreduce(const void* const* in, void* const* out, int nranks, size_t count,
                         sar_dtype dtype, sar_algo algo, sar_stream_t stream);

/*
 * sar_allreduce_accum -- the fused rsag allreduce with another accumulator
 * (mscclpp commit history, "Add mixed-precision accumulation for allreduce":
 * accumDtype, with AUTO resolving to the input type; FP8 inputs reduced in
 * float16 or float32).
 *
 * Every partial sum is rounded into `accum`:
 *   acc_0 = R_accum(f32(in[0][i])),
 *   acc_k = R_accum(f32(acc_{k-1}) + f32(in[k][i]))   (binary32 add, then RNE),
 *   out[j][i] = R_dtype(acc_{N-1}).
 * accum: SAR_FP32 (identical to sar_allreduce with SAR_ALGO_RSAG), SAR_FP16,
 * SAR_BF16, or `dtype` itself (native accumulation, e.g. e4m3fn with
 * saturation at every step).  Other values return SAR_ERR_UNSUPPORTED_DTYPE.
 * Buffers, chunking and errors as sar_allreduce.
 */
SAR_API sar_status sar_allreduce_accum(const void* const* in, void* const* out, int nranks, size_t count,
                                       sar_dtype dtype, sar_dtype accum, sar_stream_t stream);

/*
 * sar_reduce_scatter -- the rsag reduce step alone.
 * For every rank r: out[r][chunk r] = the reduced chunk (as in sar_allreduce).
 * No other element of any output is written.
 */
SAR_API sar_status sar_reduce_scatter(const void* const* in, void* const* out, int nranks, size_t count,
                              sar_dtype dtype, sar_stream_t stream);

/*
 * sar_all_gather -- the rsag write-back step alone.
 * For every rank r and every j != r: out[j][chunk r] = out[r][chunk r]
 * (a bitwise copy).  After sar_reduce_scatter this completes the allreduce.
 */
SAR_API sar_status sar_all_gather(void* const* out, int nranks, size_t count, sar_dtype dtype,
                          sar_stream_t stream);

/*
 * sar_rsag_chunk -- elements per rank chunk: ceil(count / nranks) rounded up
 * to a whole 16-byte vector of elements.  Returns 0 for invalid arguments.
 */
SAR_API size_t sar_rsag_chunk(size_t count, int nranks, sar_dtype dtype);

/*
 * sar_ll_packet_bytes -- bytes of one rank's LL packet buffer:
 * ceil(count * element size / 4) packets of 8 bytes.  0 for a bad dtype.
 *
 * Packet w of rank r (mscclpp commit history, allreduce_allpair_packet fix;
 * layout: 4-byte payload + 4-byte flag): bytes 0..3 are bytes 4w..4w+3 of
 * in[r] (zero past the end of the input), bytes 4..7 the epoch as a
 * little-endian uint32.  Each packet is written and read as one
 * single-copy-atomic 8-byte access (alone, or as an element of a 16- or
 * 32-byte vector access), so a reader that sees the flag also sees the
 * payload.
 *
 * Packet buffers belong to the caller, must be 16-byte aligned, and must be
 * zeroed once before first use: epoch 0 is reserved for "never written"
 * (mscclpp commit history, the TokenPool fix: recycled counters must not keep
 * stale values).  Epochs must not repeat while a buffer can still hold packets
 * of the earlier use; after 2^32 - 1 epochs, zero the buffers again.
 */
SAR_API size_t sar_ll_packet_bytes(size_t count, sar_dtype dtype);

/*
 * sar_ll_pack -- the LL send: rank r's whole input is written as packets to
 * pkts[r], every flag = epoch.  epoch == 0 returns SAR_ERR_INVALID_ARG.
 */
SAR_API sar_status sar_ll_pack(const void* const* in, void* const* pkts, int nranks, size_t count,
                       sar_dtype dtype, uint32_t epoch, sar_stream_t stream);

/*
 * sar_ll_unpack_reduce -- the LL reduce and write-back.
 *
 * Simulated rank r owns a 1/N chunk of the packet index range (ceil(P / N)
 * packets of the P per buffer).  For each packet in it, for k = 0..N-1 in
 * order, it loads pkts[k]'s packet, polls until the flag equals `epoch`, adds
 * the payload's elements in binary32, rounds once and stores the elements to
 * all N outputs.  The values equal sar_allreduce's.
 *
 * A poll re-reads a packet at most `max_spins` times (with a short sleep
 * between reads).  When one runs out, the kernel stores SAR_ERR_TIMEOUT into
 * *d_status (only if it still holds 0), every thread stops polling, and the
 * outputs are unspecified; the call itself has already returned SAR_OK.
 * Read the status with sar_read_device_status.
 *
 * d_status : caller-owned device int32, zeroed by the caller; it is never
 *            cleared by the library, so one word can collect the status of
 *            many calls.  max_spins == 0 returns SAR_ERR_INVALID_ARG.
 */
SAR_API sar_status sar_ll_unpack_reduce(const void* const* pkts, void* const* out, int nranks, size_t count,
                                sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                                int32_t* d_status, sar_stream_t stream);

/*
 * sar_allreduce_ll -- the LL all-pair allreduce: sar_ll_pack then
 * sar_ll_unpack_reduce with the same epoch, stream-ordered.  `pkts` is the
 * caller's packet scratch (nranks buffers of sar_ll_packet_bytes each).
 */
SAR_API sar_status sar_allreduce_ll(const void* const* in, void* const* out, void* const* pkts, int nranks,
                            size_t count, sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                            int32_t* d_status, sar_stream_t stream);

/*
 * sar_allreduce_ll_double -- sar_allreduce_ll on a double-buffered packet
 * scratch (mscclpp commit history, the allreduce_allpair_packet fix: the
 * packet scratch is used in alternating halves, so a call does not overwrite
 * packets that the previous call may still be reading).
 *
 * pkts[r] holds two halves of H = sar_ll_packet_bytes(count, dtype) rounded
 * up to a multiple of 16 bytes, so 2*H bytes, 16-byte aligned, zeroed once
 * before first use.  A call with epoch e packs into and polls half (e & 1),
 * which starts at pkts[r] + (e & 1) * H.  Two calls whose epochs have
 * different parity therefore touch disjoint packets and may run at the same
 * time, for example on two streams sharing one scratch allocation; calls
 * whose epochs have the same parity must not overlap on the GPU.  Everything
 * else (values, status, errors) as sar_allreduce_ll.
 */
SAR_API sar_status sar_allreduce_ll_double(const void* const* in, void* const* out, void* const* pkts, int nranks,
                                           size_t count, sar_dtype dtype, uint32_t epoch, uint64_t max_spins,
                                           int32_t* d_status, sar_stream_t stream);

/*
 * sar_allreduce_ll_fused -- the LL all-pair allreduce in one launch (mscclpp
 * commit history, the allreduce_allpair_packet fix: send, reduce and
 * write-back in the same thread block).  Results equal sar_allreduce_ll's,
 * and so does the packet image left in pkts.  Two forms:
 *  - up to 256 KiB per rank (count * element size), block b plays every rank
 *    for one slice of the packets: it packs the slice of every in[k] into
 *    pkts[k], polls those packets (written by other warps of the block),
 *    reduces in rank order and writes to all N outputs; no block waits for
 *    another;
 *  - above that, one cooperative launch: every block of simulated rank r
 *    packs its share of in[r] into pkts[r], then polls its share of rank r's
 *    packet chunk in all N packet buffers while other blocks are still
 *    packing.  Blocks wait on each other, so all blocks must be co-resident;
 *    a launch the device cannot make co-resident fails with SAR_ERR_CUDA.
 *
 * Epoch: with d_epoch == NULL the caller's `epoch` (non-zero, as in
 * sar_ll_pack).  Otherwise d_epoch is a caller-owned device epoch counter:
 * 8 bytes, 8-byte aligned, zeroed once before first use, read and written by
 * the kernels as one uint64 (little-endian) whose bits 20..63 count the
 * launches that used it (bits 0..19 are zero between launches).  The k-th
 * launch (k = 0, 1, ...) uses epoch (k mod (2^32 - 1)) + 1, so a launch
 * captured in a CUDA graph gets a fresh epoch on every replay; `epoch` is
 * then ignored.  To continue after host epochs 1..e, store (uint64)e << 20.
 * Every block takes the epoch with one atomic add at its start; no block
 * waits for another and nothing is written at the end of the launch.  One
 * counter must not be shared by launches that can overlap on the GPU.
 *
 * Epochs repeat every 2^32 - 1 launches of one counter.  Each launch writes
 * all of its packets with the new epoch, and consecutive launches always use
 * different epochs, so calls with one count per set of buffers never see a
 * stale packet.  A caller that varies `count` on the same buffers leaves
 * packets past the smaller calls' ends untouched; it should zero the packet
 * buffers and the counter at least once every 2^32 - 2 launches (about 2.4
 * hours of back-to-back 2 us launches), for example by counting the replays
 * of its graphs.
 *
 * Packet buffers, max_spins and d_status as in sar_ll_unpack_reduce, except
 * that the first 16 re-reads of a packet come without a sleep (the packets
 * are written by the same launch), and a thread looks at *d_status (to stop
 * when another has given up) only after them.  A poll that runs out does not
 * stop the launch from advancing the counter.
 */
SAR_API sar_status sar_allreduce_ll_fused(const void* const* in, void* const* out, void* const* pkts, int nranks,
                                          size_t count, sar_dtype dtype, uint32_t epoch, uint64_t* d_epoch,
                                          uint64_t max_spins, int32_t* d_status, sar_stream_t stream);

/*
 * sar_allreduce_ll_writeback -- the LL all-pair allreduce with the write-back
 * as a second round of flagged packets, in one launch (mscclpp
 * commit history: the allreduce_allpair_packet fix's send / reduce /
 * write-back, and the ReadPutPacket change that reads packet data once and
 * writes it to several destinations).
 *
 * As sar_allreduce_ll_fused, except that each rank's reduced chunk is written
 * as packets (flag = epoch) into the result packet buffer `res` and then
 * polled again and unpacked into the outputs:
 *   multi_dest != 0 : each result packet is read once and written to all N
 *                     outputs (by another warp of the block that reduced it
 *                     up to 1 MiB per rank, in the sliced form of
 *                     sar_allreduce_ll_fused; above, cooperatively, by the
 *                     blocks of another rank than its reducer);
 *   multi_dest == 0 : every rank reads every result packet and writes its own
 *                     output (N reads per packet; sliced up to 256 KiB per
 *                     rank, the (rank, packet group) reads spread over a
 *                     block's threads; cooperative above).
 * Results equal sar_allreduce_ll's; after the call `res` holds the packets of
 * the reduced data, zero-padded like sar_ll_pack's.
 *
 * res : caller-owned device buffer of sar_ll_packet_bytes(count, dtype) bytes,
 *       16-byte aligned, zeroed once before first use; the same epoch rules as
 *       the send packet buffers.  d_epoch: the device epoch counter as in
 *       sar_allreduce_ll_fused (one counter may serve both entry points).
 */
SAR_API sar_status sar_allreduce_ll_writeback(const void* const* in, void* const* out, void* const* pkts, void* res,
                                              int nranks, size_t count, sar_dtype dtype, uint32_t epoch,
                                              uint64_t* d_epoch, int multi_dest, uint64_t max_spins,
                                              int32_t* d_status, sar_stream_t stream);

/* Largest rank count of sar_allreduce_ll_cluster (CTAs per thread-block cluster). */
#define SAR_LL_CLUSTER_MAX_RANKS 16

/*
 * sar_allreduce_ll_cluster -- the LL all-pair allreduce with the packets
 * exchanged through distributed shared memory inside thread-block clusters
 * (mscclpp commit history, the allreduce_allpair_packet fix: each rank sends
 * its data as flag-checked packets into every peer's scratch, the peer polls
 * its own scratch, reduces and writes back, all in one thread block).
 *
 * The packet range of every rank is cut into slices of 64, 128 or 256
 * packets per rank chunk (the smallest that keeps the grid small enough: more
 * clusters for small calls, the clusters that fit at once for large ones);
 * each slice is handled by one cluster of nranks CTAs, CTA r acting for
 * simulated rank r.  CTA k packs its input words of the slice of every
 * chunk r into 8-byte packets {payload, flag} and stores them into the shared
 * memory of CTA r; CTA r polls the flags of the packets it received from all
 * ranks (bounded by max_spins re-reads per packet), adds the payloads in rank
 * order 0..N-1 in binary32, rounds once and writes the result to all N
 * outputs.  Results equal sar_allreduce's bit for bit.
 *
 * The packet slots live in each CTA's shared memory and are cleared at the
 * start of every launch (before a cluster barrier), so the call needs no
 * scratch buffer, no epoch and no state between calls: it allocates nothing,
 * a CUDA graph may replay it as it is, and calls on different streams may
 * run at the same time.  Packets never reach global memory, so the HBM
 * traffic is N*S read plus N*S written.
 *
 * nranks : 1 .. SAR_LL_CLUSTER_MAX_RANKS (16; clusters of more than 8 CTAs use
 *          the non-portable cluster size), else SAR_ERR_UNSUPPORTED_NRANKS.
 * in, out, count, dtype : as sar_allreduce (in place allowed).
 * max_spins, d_status : as sar_ll_unpack_reduce; a poll can run out only when
 *          max_spins is smaller than the time the peers' stores take.
 */
SAR_API sar_status sar_allreduce_ll_cluster(const void* const* in, void* const* out, int nranks, size_t count,
                                            sar_dtype dtype, uint64_t max_spins, int32_t* d_status,
                                            sar_stream_t stream);

/*
 * Size of the fixed LL packet scratch inside the library used by
 * sar_allreduce_ll_noalloc: 16 MiB per GPU.  A call fits when
 * nranks * (sar_ll_packet_bytes(count, dtype) rounded up to 256) is at most
 * this size, e.g. up to 1 MiB per rank with 8 ranks.
 */
#define SAR_LL_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * sar_allreduce_ll_noalloc -- sar_allreduce_ll without caller-provided packet
 * scratch, for callers that cannot allocate device memory: code inside a
 * framework whose allocator owns the device memory, plugins with a fixed
 * memory budget, or paths where a cudaMalloc would synchronise the device or
 * is not allowed.  MSCCL++ has no counterpart of this entry point.
 *
 * The outputs equal sar_allreduce_ll's bit for bit.  The call allocates
 * nothing: the packet scratch is a fixed array of SAR_LL_NOALLOC_SCRATCH_BYTES
 * (plus one status word) compiled into the library, which every GPU that
 * loads the library's device code holds until the process exits.  The caller
 * still passes the inputs and outputs.
 *
 * - Sizes beyond the array (see SAR_LL_NOALLOC_SCRATCH_BYTES) return
 *   SAR_ERR_INVALID_ARG before anything is launched.
 * - The first call on a device looks up the array's device address on that
 *   device (the current one); make that first call before any CUDA graph
 *   capture on the device.  If the lookup fails (SAR_ERR_CUDA), nothing is
 *   kept and the next call tries again.
 * - The epoch is managed by the library (a new one per call and device).
 * - d_status: an optional caller device int32 that receives SAR_ERR_TIMEOUT if
 *   a poll runs out of spins (as in sar_ll_unpack_reduce).  With NULL, an
 *   internal status word is cleared and used instead, and a timeout is not
 *   reported to the caller.
 * - Every call on a device shares the one array, which keeps the last call's
 *   packets.  Calls that overlap on the GPU (for example on two streams
 *   without ordering between them) race on it: their outputs are undefined
 *   and their polls may time out.
 */
SAR_API sar_status sar_allreduce_ll_noalloc(const void* const* in, void* const* out, int nranks,
                                            size_t count, sar_dtype dtype, uint64_t max_spins,
                                            int32_t* d_status, sar_stream_t stream);

/*
 * sar_fp8_convert -- dst[i] = R_dst(f32(src[i])) for count elements.
 *
 * Supported pairs: e4m3fn -> {fp32, fp16, bf16} (exact) and
 * {fp32, fp16, bf16} -> e4m3fn (one round-to-nearest-even, finite overflow and
 * infinities saturate to +-448, NaN stays NaN).  FP8 with higher-precision
 * accumulation: mscclpp commit history, the ROCm FP8 summary and "Add
 * mixed-precision accumulation for allreduce".  Other pairs return
 * SAR_ERR_UNSUPPORTED_DTYPE.  src and dst must not overlap.
 */
SAR_API sar_status sar_fp8_convert(const void* src, sar_dtype src_dtype, void* dst, sar_dtype dst_dtype,
                           size_t count, sar_stream_t stream);

/*
 * sar_read_device_status -- synchronises `stream`, reads *d_status and returns
 * it as a sar_status (SAR_OK or SAR_ERR_TIMEOUT), or SAR_ERR_CUDA if the copy
 * fails.  Not for use inside a CUDA graph capture.
 */
SAR_API sar_status sar_read_device_status(const int32_t* d_status, sar_stream_t stream);

/* sar_status_string -- a static, human-readable name for a status. */
SAR_API const char* sar_status_string(sar_status status);

#ifdef __cplusplus
}
#endif

#endif /* SAR_H_ */
