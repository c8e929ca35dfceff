// score_fwd_v4_fused.cu -- V4 scoring kernels, three selection groups, fused ReLU
// scoring and selection only (instantiated here, in a translation unit of their
// own, so that the configurations compile in parallel).
#include "score_fwd.cuh"

namespace lidx {

LIDX_STATUS_READER(status_score_v4_fused)

cudaError_t score_launch_v4_fused(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& ma, int smem, int grid) {
    return launch_any<false, kCfgFused>(a, mq, mk, ma, smem, grid);
}

}  // namespace lidx
