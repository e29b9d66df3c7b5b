// rsag_e4m3fn.cu -- the rsag reduce kernels for e4m3fn elements with a binary32
// accumulator (one translation unit per element type and accumulator group
// keeps the parallel build short).
#include "rsag_kernels.cuh"

namespace sar {
template cudaError_t launch_rsag_wide<SAR_FP8_E4M3FN>(RsagMode, int, const RankPtrs&, size_t, size_t, bool,
                                              cudaStream_t);
}  // namespace sar
