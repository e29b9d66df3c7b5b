// rsag_bf16.cu -- the rsag reduce kernels for bf16 elements with a binary32
// accumulator (one translation unit per element type and accumulator group
// keeps the parallel build short).
#include "rsag_kernels.cuh"

namespace sar {
template cudaError_t launch_rsag_wide<SAR_BF16>(RsagMode, int, const RankPtrs&, size_t, size_t, bool, cudaStream_t);
}  // namespace sar
