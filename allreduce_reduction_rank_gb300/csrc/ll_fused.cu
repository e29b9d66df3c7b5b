// ll_fused.cu -- sar_allreduce_ll_fused: the LL all-pair allreduce in one
// launch, with the result written back directly from registers (the kernels,
// their phases and the choice between them are described in ll_coop.cuh).
#include "ll_coop.cuh"

namespace sar {

cudaError_t launch_ll_fused(sar_dtype dt, int nranks, const RankPtrs& data, void* const* pkts, size_t count,
                            uint32_t epoch, uint64_t* ctrl, uint64_t max_spins, int32_t* status, bool in16,
                            bool out16, cudaStream_t stream) {
    return llc::coop_launch<llc::kDirect>(dt, nranks, data, pkts, nullptr, count, epoch, ctrl, max_spins, status,
                                          in16, out16, stream);
}

}  // namespace sar
