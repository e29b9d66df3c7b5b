// rsag_e4m3fn_acc.cu -- the fused rsag kernels for e4m3fn elements with fp16, bf16
// or native accumulation.
#include "rsag_kernels.cuh"

namespace sar {
template cudaError_t launch_rsag_narrow<SAR_FP8_E4M3FN>(sar_dtype, int, const RankPtrs&, size_t, size_t, bool,
                                              cudaStream_t);
}  // namespace sar
