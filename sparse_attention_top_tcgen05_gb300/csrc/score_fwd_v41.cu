// score_fwd_v41.cu -- V4.1 scoring kernels (instantiated here, in a
// translation unit of their own, so that the configurations compile in parallel).
#include "score_fwd.cuh"

namespace lidx {

LIDX_STATUS_READER(status_score_v41)

cudaError_t score_launch_v41(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& ma, int smem, int grid) {
    return launch_any<true, kCfgAll>(a, mq, mk, ma, smem, grid);
}

}  // namespace lidx
