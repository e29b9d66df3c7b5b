// sar_internal.h -- launchers between the C ABI (sar_api.cu) and the kernels.
// All arguments have been validated by the caller.
#pragma once

#include <cstddef>
#include <cstdint>

#include <utility>

#include <cuda_runtime.h>

#include "../../include/sar.h"

namespace sar {

// Kernel launch with programmatic stream serialization: the kernel may be
// scheduled before the previous kernel in the stream has finished, and waits
// for it with pdl_wait() (sar_device.cuh) before touching memory, so the
// results are those of plain stream order.  Measured on GB300 against plain
// launches (interleaved runs): faster at every size, e.g. 2 x 16 MiB bf16
// 8.2 -> 6.1 us per call eager and 6.4 -> 6.0 us in a CUDA graph, 8 x 64 MiB
// fp16 155.8 -> 153.2 us eager.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// What an rsag launch writes: the fused allreduce writes the reduced chunk to
// every output; the reduce-scatter step writes it to the owning rank only.
enum RsagMode { kFused = 0, kReduceScatter = 1 };

struct RankPtrs {
    const void* in[SAR_MAX_RANKS];
    void* out[SAR_MAX_RANKS];
};

// rsag reduce (fused or reduce-scatter).  `vec` selects 16-byte vectors
// (every buffer 16-byte aligned).
cudaError_t launch_rsag(RsagMode mode, sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                        size_t chunk, bool vec, cudaStream_t stream);

// Fused rsag allreduce with partial sums rounded into `acc` (fp16, bf16, or
// e4m3fn for e4m3fn inputs).
cudaError_t launch_rsag_accum(sar_dtype dt, sar_dtype acc, int nranks, const RankPtrs& p, size_t count,
                              size_t chunk, bool vec, cudaStream_t stream);

// The reduce launchers of one element type (rsag_kernels.cuh): binary32
// accumulation in either mode (instantiated in rsag_<type>.cu), and fp16 /
// bf16 / native FP8 accumulation in the fused mode (rsag_<type>_acc.cu).
template <int DT>
cudaError_t launch_rsag_wide(RsagMode mode, int nranks, const RankPtrs& p, size_t count, size_t chunk, bool vec,
                             cudaStream_t s);
template <int DT>
cudaError_t launch_rsag_narrow(sar_dtype acc, int nranks, const RankPtrs& p, size_t count, size_t chunk, bool vec,
                               cudaStream_t s);

// rsag all-gather: out[j][chunk r] = out[r][chunk r], j != r (bytes).
cudaError_t launch_all_gather(int nranks, const RankPtrs& p, size_t count, size_t esize,
                              size_t chunk, bool vec, cudaStream_t stream);

// LL pack: pkts[r] <- packets of in[r] (p.out holds the packet buffers).
cudaError_t launch_ll_pack(int nranks, const RankPtrs& p, size_t bytes, uint32_t epoch,
                           bool vec, cudaStream_t stream);

// LL poll + unpack + reduce + write-back (p.in holds the packet buffers).
cudaError_t launch_ll_unpack_reduce(sar_dtype dt, int nranks, const RankPtrs& p, size_t count,
                                    uint32_t epoch, uint64_t max_spins, int32_t* status,
                                    bool vec_out, cudaStream_t stream);

// LL send + reduce + write-back in one cooperative launch.  ctrl: optional
// device epoch counter (launches << 20); with it the k-th launch uses epoch
// (k mod (2^32 - 1)) + 1.
cudaError_t launch_ll_fused(sar_dtype dt, int nranks, const RankPtrs& data, void* const* pkts, size_t count,
                            uint32_t epoch, uint64_t* ctrl, uint64_t max_spins, int32_t* status, bool in16,
                            bool out16, cudaStream_t stream);

// LL with the write-back as a second packet round into `res`; multi_dest:
// each result packet is read once and written to all outputs.
cudaError_t launch_ll_writeback(sar_dtype dt, int nranks, const RankPtrs& data, void* const* pkts, void* res,
                                size_t count, uint32_t epoch, uint64_t* ctrl, bool multi_dest, uint64_t max_spins,
                                int32_t* status, bool in16, bool out16, cudaStream_t stream);

// Test support for the fixed scratch (not exported from the library; a test
// program links the object files): sets the last epoch used on `dev` and
// returns the array's device address there (nullptr if it was not looked up).
unsigned char* testing_fixed_scratch(int dev, bool set_epoch, uint32_t last_epoch);

// LL through distributed shared memory: one cluster of nranks CTAs per slice
// (ll_cluster.cu); nranks <= SAR_LL_CLUSTER_MAX_RANKS.
cudaError_t launch_ll_cluster(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                              int32_t* status, bool in16, bool out16, cudaStream_t stream);

// LL of a small call inside one CTA, every rank's packets in its shared
// memory (ll_cta.cu); the slots take ll_cta_slot_bytes(), at most
// kLLCtaMaxSlotBytes.
constexpr size_t kLLCtaMaxSlotBytes = size_t(64) << 10;
size_t ll_cta_slot_bytes(int nranks, size_t count, sar_dtype dt);
cudaError_t launch_ll_cta(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                          int32_t* status, bool in16, bool out16, cudaStream_t stream);
// The same over a grid: CTA b plays every rank for one slice of the packets
// (ll_cta.cu); any size, no scratch.
cudaError_t launch_ll_slice(sar_dtype dt, int nranks, const RankPtrs& p, size_t count, uint64_t max_spins,
                            int32_t* status, bool in16, bool out16, cudaStream_t stream);

cudaError_t launch_convert(const void* src, sar_dtype src_dt, void* dst, sar_dtype dst_dt,
                           size_t count, bool vec, cudaStream_t stream);

size_t esize_of(sar_dtype dt);

}  // namespace sar
