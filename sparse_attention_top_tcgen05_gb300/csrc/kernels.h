// kernels.h -- internal interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lidx {

// V4 scoring (+ optional fused top-k) kernel parameters.
struct ScoreParams {
    int B, S, Skv, H, D, ratio, act;
    const int32_t* ks;  // nullable with ke: causal ranges from ratio
    const int32_t* ke;
    const float* w;     // [S,B,H]
    float* logits;      // nullable: [B,S,Skv]
    int clean;
    float* scratch;     // per-CTA row buffers when logits == nullptr and topk > 0
    int64_t scratch_stride_cta;
    int topk;           // 0: no selection
    int32_t* out_idx;   // [B,S,topk]
    float* out_sc;      // [B,S,topk]
    // V4.1 (BSHD layouts, bf16 weights and scores, explicit visibility)
    const uint16_t* w16;      // [B,S,H] bf16
    const uint8_t* allowed;   // [B,S,Skv]
    uint16_t* out16;          // [B,S,Skv] bf16
    uint8_t* tilemap;         // [B, qtiles, ntk]: 1 where the block has a visible pair (written by the kernel)
    int2* urange;             // nullable [B, qtiles]: key tiles [x, y) holding each query tile's visible
                              // pairs (written by the kernel; (0, 0) when there are none)
    int ntk;                  // key tiles per row
    int vis_tma;              // 1: visibility flags staged by TMA (set by the launcher)
    const int32_t* idx_in;    // nullable [B,S,topk]: score these keys instead of selecting
    uint64_t wait_ns;         // limit of every pipeline wait
    int debug_stall;          // 1: the TMA producer issues nothing (failure-detection tests)
    int warp_rows;            // 1: each selection warp selects rows of its own (short rows)
    // filled by the launcher
    int num_units, qtiles, Skv_pad, swz;
};

struct ScoreLaunch {
    ScoreParams p;
    const void* q;
    const void* k;
    void* stream;
    int num_sms;
    int launched;
};

// cuTensorMapEncodeTiled through the runtime's driver entry point; returns 0 on success.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* addr,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                 const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle);

int score_fwd_launch(ScoreLaunch& a);
// the scoring kernels of one configuration for the call's head count
cudaError_t score_launch_v4(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& ma, int smem, int grid);
cudaError_t score_launch_v4_short(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& ma, int smem, int grid);
cudaError_t score_launch_v4_fused(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& ma, int smem, int grid);
cudaError_t score_launch_v41(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& ma, int smem, int grid);
int score_v41_launch(ScoreLaunch& a);
int score_query_tile(int H);  // query rows per tile for H heads
size_t score_scratch_bytes(int64_t S, int64_t Skv, int H, int num_sms);

cudaError_t extract_launch(const float* logits, const int32_t* idx, int64_t rows, int64_t Skv,
                           int topk, float* out, cudaStream_t stream);

cudaError_t topk_rows_launch(const float* logits, int64_t rows, int S, int Skv, int ratio,
                             const int32_t* ks, const int32_t* ke, int topk, int32_t* out_idx,
                             float* out_sc, cudaStream_t stream);
// selection over bf16 rows; -inf entries are not candidates (V4.1 scores)
cudaError_t topk_rows_bf16_launch(const uint16_t* scores, int64_t rows, int S, int Skv, const int2* urange,
                                  int QT, int topk, int32_t* out_idx, uint16_t* out_sc, cudaStream_t stream);
// backward through the selected entries (bwd.cu)
struct BwdLaunch {
    const void* q;
    const void* k;
    const float* w;
    const int32_t* idx;
    const float* grad;
    int B, S, Skv, H, D, ratio, topk, act, grad_dtype;
    const int32_t* ks;  // nullable with ke: causal ranges from ratio
    const int32_t* ke;
    void* dq;           // fp32 or bf16 (grad_dtype)
    void* dk;
    float* dw;
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
    int num_sms;
};
cudaError_t bwd_launch(const BwdLaunch& a);
size_t bwd_workspace_bytes(int64_t B, int64_t S, int64_t Skv, int H, int D, int topk, int num_sms);

cudaError_t pad_launch(int64_t n, int32_t* idx, float* sc, cudaStream_t stream);
// padding with bf16 scores; and given indices copied with -inf scores
cudaError_t pad16_launch(int64_t n, int32_t* idx, uint16_t* sc, cudaStream_t stream);
cudaError_t copy_pad_launch(int64_t n, const int32_t* in, int32_t* idx, float* sc, cudaStream_t stream);

// argument rules of the V4 forward that need no device (api.cu); LIDX_OK or an error
int check_fwd(const void* q, const void* k, const float* w, int64_t B, int64_t S, int64_t Skv, int H,
              int D, int compress_ratio, const int32_t* ks, const int32_t* ke, int topk, int act,
              const int32_t* topk_indices_in, const float* logits_out, const int32_t* indices_out,
              const float* scores_out);

// host-side state shared by the launchers (api.cu)
int current_sms();                                   // SM count of the current device
cudaError_t set_smem_attr(const void* fn, int smem);  // once per (device, kernel, size)
uint64_t wait_limit_ns();                             // limit of every pipeline wait
int debug_stall();                                    // failure-detection test switch

// per-TU status readers (see LIDX_STATUS_READER): value, or -1 on a CUDA error
int status_score_v4(int clear);        // status words of the scoring kernels' units
int status_score_v4_short(int clear);
int status_score_v4_fused(int clear);
int status_score_v41(int clear);
int status_misc(int clear);
int status_bwd(int clear);

}  // namespace lidx
