// rsag_fp16_acc.cu -- the fused rsag kernels for fp16 elements with fp16, bf16
// or native accumulation.
#include "rsag_kernels.cuh"

namespace sar {
template cudaError_t launch_rsag_narrow<SAR_FP16>(sar_dtype, int, const RankPtrs&, size_t, size_t, bool, cudaStream_t);
}  // namespace sar
