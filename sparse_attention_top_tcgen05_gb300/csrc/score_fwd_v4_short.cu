// score_fwd_v4_short.cu -- V4 scoring kernels, six selection groups for rows of at most 1024 keys (instantiated here, in a
// translation unit of their own, so that the configurations compile in parallel).
#include "score_fwd.cuh"

namespace lidx {

LIDX_STATUS_READER(status_score_v4_short)

cudaError_t score_launch_v4_short(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& ma, int smem, int grid) {
    return launch_any<false, kCfgShort>(a, mq, mk, ma, smem, grid);
}

}  // namespace lidx
