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
    const uint8_t* tilemap;   // [B, qtiles, ntk]: 1 where the block has a visible pair
    int ntk;                  // key tiles per row
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
int score_v41_launch(ScoreLaunch& a);
int score_query_tile(int H);  // query rows per tile for H heads
cudaError_t v41_mask_launch(const uint8_t* allowed, uint16_t* out, uint8_t* tilemap, int B, int S,
                            int Skv, int QT, cudaStream_t stream);
size_t score_scratch_bytes(int64_t S, int64_t Skv, int H, int num_sms);

cudaError_t extract_launch(const float* logits, const int32_t* idx, int64_t rows, int64_t Skv,
                           int topk, float* out, cudaStream_t stream);

cudaError_t topk_rows_launch(const float* logits, int64_t rows, int S, int Skv, int ratio,
                             const int32_t* ks, const int32_t* ke, int topk, int32_t* out_idx,
                             float* out_sc, cudaStream_t stream);
// backward through the selected entries (bwd.cu)
struct BwdLaunch {
    const void* q;
    const void* k;
    const float* w;
    const int32_t* idx;
    const float* grad;
    int B, S, Skv, H, D, ratio, topk, act;
    float* dq;
    float* dk;
    float* dw;
    cudaStream_t stream;
    int num_sms;
};
cudaError_t bwd_launch(const BwdLaunch& a);

// forward with given indices (gather.cu)
struct GatherLaunch {
    const void* q;
    const void* k;
    const float* w;
    const int32_t* idx;
    int B, S, Skv, H, D, ratio, topk, act;
    int32_t* out_idx;
    float* out_sc;
    cudaStream_t stream;
    int num_sms;
};
cudaError_t gather_launch(const GatherLaunch& a);

cudaError_t pad_launch(int64_t n, int32_t* idx, float* sc, cudaStream_t stream);

// per-TU status readers (see LIDX_STATUS_READER): value, or -1 on a CUDA error
int status_score_fwd(int clear);
int status_misc(int clear);

}  // namespace lidx
