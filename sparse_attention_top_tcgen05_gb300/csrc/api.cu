// api.cu -- the C ABI of liblidx.so (declared in include/lidx.h): argument
// validation, tensor-map encoding and kernel launches on the caller's stream.
// No device memory is allocated here; buffers belong to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "lidx.h"
#include "kernels.h"
#include "topk.cuh"

namespace lidx {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* addr,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                 const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = get_encode();
    if (!fn) return 1;
    CUresult r = fn(map, dtype, (cuuint32_t)rank, addr, dims, strides_bytes, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

// SM count of the current device, 0 if it is not an sm_103 part.
static int device_sms(bool require_sm103) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (require_sm103 && !(major == 10 && minor == 3)) return 0;
    return sms;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool pow2_heads(int H) { return H >= 1 && H <= 128 && (H & (H - 1)) == 0; }

// Shared shape rules of the scoring calls (heads a power of two <= 128,
// index_dim a multiple of 16: "deepseek_v41.indexer" page, queries parameter).
static int check_dims(int64_t B, int64_t S, int64_t Skv, int H, int D) {
    if (B < 1 || S < 1 || Skv < 0) return LIDX_ERR_SHAPE;
    if (!pow2_heads(H) || D < 16 || D % 16 != 0 || D > 128) return LIDX_ERR_SHAPE;
    if (S > (1 << 30) || Skv > (1 << 30) || B > (1 << 20)) return LIDX_ERR_SHAPE;
    return LIDX_OK;
}

}  // namespace lidx

using namespace lidx;

extern "C" {

int lidx_version(void) { return 0x000100; }

const char* lidx_status_string(int status) {
    switch (status) {
        case LIDX_OK: return "ok";
        case LIDX_ERR_NULL: return "a required pointer is NULL";
        case LIDX_ERR_SHAPE: return "a size or shape rule is violated";
        case LIDX_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
        case LIDX_ERR_UNSUPPORTED: return "request is outside what this build implements";
        case LIDX_ERR_WORKSPACE: return "workspace is missing or too small";
        case LIDX_ERR_CUDA: return "a CUDA call failed";
        case LIDX_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on its pipeline";
        case LIDX_ERR_NO_DEVICE: return "no sm_103 device is current";
        default: return "unknown status";
    }
}

size_t lidx_workspace_bytes(int op, int64_t B, int64_t S, int64_t Skv, int H, int D, int topk,
                            int logits_materialised) {
    (void)B;
    (void)D;
    int sms = device_sms(false);
    if (sms <= 0) sms = 256;  // no device: an upper bound
    if (op == LIDX_OP_INDEXER_FWD) {
        if (logits_materialised || topk <= 0 || !pow2_heads(H)) return 0;
        return score_scratch_bytes(S, Skv, H, sms);
    }
    if (op == LIDX_OP_SCORES_V41) {
        // one byte per (batch, query tile, 128-key tile): the visibility tile map
        if (!pow2_heads(H) || Skv <= 0 || B <= 0 || S <= 0) return 0;
        const int64_t QT = score_query_tile(H);
        const int64_t bytes = B * ((S + QT - 1) / QT) * ((Skv + 127) / 128);
        return (size_t)((bytes + 255) / 256 * 256);
    }
    return 0;
}

int lidx_device_status(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LIDX_ERR_CUDA;
    int a = status_score_fwd(1), b = status_misc(1);
    if (a < 0 || b < 0) return LIDX_ERR_CUDA;
    if (a) return a;
    return b;
}

int lidx_indexer_fwd(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                     int64_t Skv, int H, int D, int compress_ratio, int topk, int act,
                     const int32_t* topk_indices_in, float* logits_out, int32_t* indices_out,
                     float* scores_out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || (!k && Skv > 0) || !w || !indices_out || !scores_out) return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if (compress_ratio < 1 || topk < 1 || topk > (1 << 20) || (act != 0 && act != 1))
        return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || (logits_out && !aligned16(logits_out)))
        return LIDX_ERR_ALIGN;
    if (topk_indices_in && !aligned16(topk_indices_in)) return LIDX_ERR_ALIGN;
    if (!topk_indices_in && Skv > kTopkCandMax) return LIDX_ERR_UNSUPPORTED;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    if (topk_indices_in && Skv > 0) {
        // given indices: no selection, score exactly those pairs
        cudaStream_t st = (cudaStream_t)stream;
        if (logits_out) {
            // logits were asked for: sweep them, then gather (masked entries are -inf)
            const int rc2 = lidx_indexer_logits(q, k, w, B, S, Skv, H, D, compress_ratio, nullptr,
                                                nullptr, 1, act, logits_out, stream);
            if (rc2) return rc2;
            if (extract_launch(logits_out, topk_indices_in, B * S, Skv, topk, scores_out, st) !=
                    cudaSuccess ||
                cudaMemcpyAsync(indices_out, topk_indices_in, sizeof(int32_t) * (size_t)(B * S * topk),
                                cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return LIDX_ERR_CUDA;
            return LIDX_OK;
        }
        GatherLaunch g;
        g.q = q;
        g.k = k;
        g.w = w;
        g.idx = topk_indices_in;
        g.B = (int)B;
        g.S = (int)S;
        g.Skv = (int)Skv;
        g.H = H;
        g.D = D;
        g.ratio = compress_ratio;
        g.topk = topk;
        g.act = act;
        g.out_idx = indices_out;
        g.out_sc = scores_out;
        g.stream = st;
        g.num_sms = sms;
        return gather_launch(g) == cudaSuccess ? LIDX_OK : LIDX_ERR_CUDA;
    }
    if (Skv == 0)  // no keys at all: every row is padding, logits has no entries
        return pad_launch(B * S * (int64_t)topk, indices_out, scores_out, (cudaStream_t)stream) ==
                       cudaSuccess
                   ? LIDX_OK
                   : LIDX_ERR_CUDA;
    ScoreLaunch a;
    memset(&a, 0, sizeof a);
    a.p.B = (int)B;
    a.p.S = (int)S;
    a.p.Skv = (int)Skv;
    a.p.H = H;
    a.p.D = D;
    a.p.ratio = compress_ratio;
    a.p.act = act;
    a.p.w = w;
    a.p.logits = logits_out;
    a.p.clean = 1;
    a.p.topk = topk;
    a.p.out_idx = indices_out;
    a.p.out_sc = scores_out;
    if (!logits_out) {
        const size_t need = score_scratch_bytes(S, Skv, H, sms);
        if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
            return LIDX_ERR_WORKSPACE;
        a.p.scratch = (float*)workspace;
    }
    a.q = q;
    a.k = k;
    a.stream = stream;
    a.num_sms = sms;
    return score_fwd_launch(a) == 0 ? LIDX_OK : LIDX_ERR_CUDA;
}

int lidx_indexer_logits(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                        int64_t Skv, int H, int D, int compress_ratio, const int32_t* ks,
                        const int32_t* ke, int clean, int act, float* logits_out, void* stream) {
    if (!q || !w || (Skv > 0 && (!k || !logits_out))) return LIDX_ERR_NULL;
    if ((ks == nullptr) != (ke == nullptr)) return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if (Skv == 0) return LIDX_OK;  // empty output
    if ((!ks && compress_ratio < 1) || (act != 0 && act != 1)) return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || !aligned16(logits_out))
        return LIDX_ERR_ALIGN;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    ScoreLaunch a;
    memset(&a, 0, sizeof a);
    a.p.B = (int)B;
    a.p.S = (int)S;
    a.p.Skv = (int)Skv;
    a.p.H = H;
    a.p.D = D;
    a.p.ratio = compress_ratio < 1 ? 1 : compress_ratio;
    a.p.act = act;
    a.p.ks = ks;
    a.p.ke = ke;
    a.p.w = w;
    a.p.logits = logits_out;
    a.p.clean = clean ? 1 : 0;
    a.q = q;
    a.k = k;
    a.stream = stream;
    a.num_sms = sms;
    return score_fwd_launch(a) == 0 ? LIDX_OK : LIDX_ERR_CUDA;
}

int lidx_extract_topk_scores(const float* logits, const int32_t* idx, int64_t B, int64_t S,
                             int64_t Skv, int topk, float* scores_out, void* stream) {
    if (!logits || !idx || !scores_out) return LIDX_ERR_NULL;
    if (B < 1 || S < 1 || Skv < 0 || topk < 1) return LIDX_ERR_SHAPE;
    if (device_sms(true) <= 0) return LIDX_ERR_NO_DEVICE;
    return extract_launch(logits, idx, B * S, Skv, topk, scores_out, (cudaStream_t)stream) ==
                   cudaSuccess
               ? LIDX_OK
               : LIDX_ERR_CUDA;
}

int lidx_topk_rows(const float* logits, int64_t rows, int64_t S, int64_t Skv, int compress_ratio,
                   const int32_t* ks, const int32_t* ke, int topk, int32_t* indices_out,
                   float* scores_out, void* stream) {
    if ((!logits && rows * Skv > 0) || !indices_out || !scores_out) return LIDX_ERR_NULL;
    if ((ks == nullptr) != (ke == nullptr)) return LIDX_ERR_NULL;
    if (rows < 0 || S < 1 || Skv < 0 || topk < 1 || topk > (1 << 20) || (!ks && compress_ratio < 1) ||
        S > (1 << 30) || Skv > (1 << 30))
        return LIDX_ERR_SHAPE;
    if (Skv > kTopkCandMax) return LIDX_ERR_UNSUPPORTED;
    if (device_sms(true) <= 0) return LIDX_ERR_NO_DEVICE;
    if (Skv == 0)
        return pad_launch(rows * (int64_t)topk, indices_out, scores_out, (cudaStream_t)stream) ==
                       cudaSuccess
                   ? LIDX_OK
                   : LIDX_ERR_CUDA;
    return topk_rows_launch(logits, rows, (int)S, (int)Skv, compress_ratio < 1 ? 1 : compress_ratio,
                            ks, ke, topk, indices_out, scores_out, (cudaStream_t)stream) == cudaSuccess
               ? LIDX_OK
               : LIDX_ERR_CUDA;
}

int lidx_indexer_scores_v41(const void* q, const void* k, const void* w, const uint8_t* allowed,
                            int64_t B, int64_t S, int64_t Skv, int H, int D, int act,
                            void* scores_out, void* workspace, size_t workspace_bytes,
                            void* stream) {
    if (!q || !w || (Skv > 0 && (!k || !allowed || !scores_out))) return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if (act != 0 && act != 1) return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || ((uintptr_t)scores_out & 1u))
        return LIDX_ERR_ALIGN;
    if (Skv == 0) return LIDX_OK;  // empty output
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    const size_t need = lidx_workspace_bytes(LIDX_OP_SCORES_V41, B, S, Skv, H, D, 0, 0);
    if (!workspace || workspace_bytes < need) return LIDX_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    // 1. visibility pass: tile map + -inf for blocks with no visible pair
    if (v41_mask_launch(allowed, (uint16_t*)scores_out, (uint8_t*)workspace, (int)B, (int)S,
                        (int)Skv, score_query_tile(H), st) != cudaSuccess)
        return LIDX_ERR_CUDA;
    // 2. tensor-core pass over the blocks with work
    ScoreLaunch a;
    memset(&a, 0, sizeof a);
    a.p.B = (int)B;
    a.p.S = (int)S;
    a.p.Skv = (int)Skv;
    a.p.H = H;
    a.p.D = D;
    a.p.ratio = 1;
    a.p.act = act;
    a.p.w16 = (const uint16_t*)w;
    a.p.allowed = allowed;
    a.p.out16 = (uint16_t*)scores_out;
    a.p.tilemap = (const uint8_t*)workspace;
    a.q = q;
    a.k = k;
    a.stream = stream;
    a.num_sms = sms;
    return score_v41_launch(a) == 0 ? LIDX_OK : LIDX_ERR_CUDA;
}

int lidx_indexer_bwd(const void* q, const void* k, const float* w, const int32_t* idx,
                     const float* grad_scores, int64_t B, int64_t S, int64_t Skv, int H, int D,
                     int compress_ratio, int topk, int act, int grad_dtype, void* dq, void* dk,
                     float* dw, void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!q || !w || !idx || !grad_scores || !dq || !dw || (Skv > 0 && (!k || !dk)))
        return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if (topk < 1 || topk > (1 << 20) || compress_ratio < 1 || (act != 0 && act != 1))
        return LIDX_ERR_SHAPE;
    if (grad_dtype != 0) return LIDX_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dw))
        return LIDX_ERR_ALIGN;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    BwdLaunch a;
    a.q = q;
    a.k = k;
    a.w = w;
    a.idx = idx;
    a.grad = grad_scores;
    a.B = (int)B;
    a.S = (int)S;
    a.Skv = (int)Skv;
    a.H = H;
    a.D = D;
    a.ratio = compress_ratio;
    a.topk = topk;
    a.act = act;
    a.dq = (float*)dq;
    a.dk = (float*)dk;
    a.dw = dw;
    a.stream = (cudaStream_t)stream;
    a.num_sms = sms;
    return bwd_launch(a) == cudaSuccess ? LIDX_OK : LIDX_ERR_CUDA;
}

}  // extern "C"
