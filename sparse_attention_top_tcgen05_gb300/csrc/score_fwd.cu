// score_fwd.cu -- host side of the scoring kernels (score_fwd.cuh): launch
// plans, tensor maps, and the choice of kernel configuration for a call.
#include "score_fwd.cuh"

namespace lidx {

// ------------------------------------------------------------------- host

static int encode_maps(const ScoreLaunch& a, CUtensorMap* mq, CUtensorMap* mk) {
    const int swz = a.p.swz, KB = swz / 2;
    const CUtensorMapSwizzle sw = swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    const int H = a.p.H, D = a.p.D, B = a.p.B;
    const int QT = kN / H;
    // q [S,B,H,D]: dims (D, H, B, S)
    cuuint64_t qdim[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B, (cuuint64_t)a.p.S};
    cuuint64_t qstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)B * H * D * 2};
    cuuint32_t qbox[4] = {(cuuint32_t)KB, (cuuint32_t)H, 1, (cuuint32_t)QT};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode_tiled(mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)a.q, qdim, qstr, qbox, es, sw))
        return 1;
    // k [Skv,B,D]: dims (D, B, Skv)
    cuuint64_t kdim[3] = {(cuuint64_t)D, (cuuint64_t)B, (cuuint64_t)(a.p.Skv > 0 ? a.p.Skv : 1)};
    cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)B * D * 2};
    cuuint32_t kbox[3] = {(cuuint32_t)KB, 1, (cuuint32_t)kM};
    if (encode_tiled(mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.k, kdim, kstr, kbox, es, sw))
        return 1;
    return 0;
}

int score_query_tile(int H) { return kN / H; }

size_t score_scratch_bytes(int64_t S, int64_t Skv, int H, int num_sms) {
    (void)S;
    const int QT = kN / H;
    const int64_t Skv_pad = (Skv + kM - 1) / kM * kM;
    return (size_t)num_sms * 2 * QT * Skv_pad * sizeof(float);  // two row buffers per CTA
}

int score_fwd_launch(ScoreLaunch& a) {
    ScoreParams& p = a.p;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = debug_stall();
    // rows of at most kTopkShort keys: each selection warp takes rows of its own
    p.warp_rows = (p.idx_in == nullptr && p.Skv <= kTopkShort) ? 1 : 0;
    const int QT = kN / p.H;
    p.swz = (p.D % 64 == 0) ? 128 : (p.D % 32 == 0 ? 64 : 32);
    p.qtiles = (p.S + QT - 1) / QT;
    p.num_units = p.B * p.qtiles;
    p.Skv_pad = (p.Skv + kM - 1) / kM * kM;
    p.scratch_stride_cta = (int64_t)QT * p.Skv_pad;
    const int grid = p.num_units < a.num_sms ? p.num_units : a.num_sms;
    if (grid <= 0) return 0;
    CUtensorMap mq, mk;
    if (encode_maps(a, &mq, &mk)) return -1;
    // at least 120 KB so that one CTA (and its 512 TMEM columns) owns each SM
    int smem = (int)smem_layout(p.D).total;
    if (smem < 120 * 1024) smem = 120 * 1024;
    if (p.H < 1 || p.H > 128 || (p.H & (p.H - 1))) return -2;
    CUtensorMap unused;
    memset(&unused, 0, sizeof unused);
    // rows of at most kTopkShortCap keys: more selection groups with smaller windows;
    // the fused-only configuration when the call asks for nothing more; else the
    // general one
    const bool plain = p.idx_in == nullptr && !p.warp_rows && p.act == 0;
    const bool short_rows = plain && p.Skv <= kTopkShortCap;
    const bool fused_only = plain && p.logits == nullptr && p.topk > 0 && p.D == 128;
    const cudaError_t e = short_rows   ? score_launch_v4_short(a, mq, mk, unused, smem, grid)
                          : fused_only ? score_launch_v4_fused(a, mq, mk, unused, smem, grid)
                                       : score_launch_v4(a, mq, mk, unused, smem, grid);
    a.launched = grid;
    return e == cudaSuccess ? 0 : -1;
}

// V4.1: q [B,S,H,D], k [B,Skv,D], allowed [B,S,Skv].  One launch: the kernel's
// visibility warps read `allowed` and build each unit's record and tile map row
// (p.tilemap, caller workspace) ahead of the tensor-core sweep.
int score_v41_launch(ScoreLaunch& a) {
    ScoreParams& p = a.p;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = debug_stall();
    if (p.H < 1 || p.H > 128 || (p.H & (p.H - 1))) return -2;
    const int QT = kN / p.H;
    p.swz = (p.D % 64 == 0) ? 128 : (p.D % 32 == 0 ? 64 : 32);
    p.qtiles = (p.S + QT - 1) / QT;
    p.num_units = p.B * p.qtiles;
    p.Skv_pad = (p.Skv + kM - 1) / kM * kM;
    p.ntk = (p.Skv + kM - 1) / kM;
    const int grid = p.num_units < a.num_sms ? p.num_units : a.num_sms;
    if (grid <= 0) return 0;
    const int swz = p.swz, KB = swz / 2;
    const CUtensorMapSwizzle sw = swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    const int H = p.H, D = p.D, B = p.B;
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUtensorMap mq, mk;
    cuuint64_t qdim[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)p.S, (cuuint64_t)B};
    cuuint64_t qstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)p.S * H * D * 2};
    cuuint32_t qbox[4] = {(cuuint32_t)KB, (cuuint32_t)H, (cuuint32_t)QT, 1};
    if (encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)a.q, qdim, qstr, qbox, es, sw))
        return -1;
    cuuint64_t kdim[3] = {(cuuint64_t)D, (cuuint64_t)p.Skv, (cuuint64_t)B};
    cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Skv * D * 2};
    cuuint32_t kbox[3] = {(cuuint32_t)KB, (cuuint32_t)kM, 1};
    if (encode_tiled(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.k, kdim, kstr, kbox, es, sw))
        return -1;
    // visibility flags by TMA: rows of `allowed` 16-byte aligned, QT <= 32 (H >= 8)
    CUtensorMap ma;
    memset(&ma, 0, sizeof ma);
    p.vis_tma = 0;
    if (QT <= 32 && (p.Skv % 16) == 0 && ((uintptr_t)p.allowed & 15) == 0) {
        cuuint64_t adim[3] = {(cuuint64_t)p.Skv, (cuuint64_t)p.S, (cuuint64_t)B};
        cuuint64_t astr[2] = {(cuuint64_t)p.Skv, (cuuint64_t)p.S * p.Skv};
        cuuint32_t abox[3] = {(cuuint32_t)kM, (cuuint32_t)QT, 1};
        if (encode_tiled(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, (void*)p.allowed, adim, astr, abox, es,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return -1;
        p.vis_tma = 1;
    }
    int smem = (int)smem_layout(p.D).total;
    if (smem < 120 * 1024) smem = 120 * 1024;
    const cudaError_t e = score_launch_v41(a, mq, mk, ma, smem, grid);
    a.launched = grid;
    return e == cudaSuccess ? 0 : -1;
}

}  // namespace lidx
