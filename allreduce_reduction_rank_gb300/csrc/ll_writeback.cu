// ll_writeback.cu -- sar_allreduce_ll_writeback: the LL all-pair allreduce
// whose write-back is a second round of flagged packets (the kernel and its
// phases are described in ll_coop.cuh).
#include "ll_coop.cuh"

namespace sar {

cudaError_t launch_ll_writeback(sar_dtype dt, int nranks, const RankPtrs& data, void* const* pkts, void* res,
                                size_t count, uint32_t epoch, uint64_t* ctrl, bool multi_dest, uint64_t max_spins,
                                int32_t* status, bool in16, bool out16, cudaStream_t stream) {
    if (multi_dest)
        return llc::coop_launch<llc::kPacketsAll>(dt, nranks, data, pkts, res, count, epoch, ctrl, max_spins, status,
                                                  in16, out16, stream);
    return llc::coop_launch<llc::kPacketsOwn>(dt, nranks, data, pkts, res, count, epoch, ctrl, max_spins, status, in16,
                                              out16, stream);
}

}  // namespace sar
