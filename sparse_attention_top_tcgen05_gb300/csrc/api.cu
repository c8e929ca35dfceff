// api.cu -- the C ABI of liblidx.so (declared in include/lidx.h): argument
// validation, tensor-map encoding and kernel launches on the caller's stream.
// No device memory is allocated here; buffers belong to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <climits>
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

// A small cache of encoded tensor maps keyed by every encode argument, so that
// repeated calls on the same buffers skip the driver's encode.
struct MapKey {
    void* addr;
    int dtype, rank, swizzle;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], es[5];
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint64_t used;
};
constexpr int kMapCache = 32;
static MapEntry g_maps[kMapCache];
static int g_nmaps = 0;
static uint64_t g_map_clock = 0;
static std::mutex g_map_mu;

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* addr,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                 const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle) {
    if (rank < 1 || rank > 5) return 1;
    MapKey k;
    memset(&k, 0, sizeof k);
    k.addr = addr;
    k.dtype = (int)dtype;
    k.rank = rank;
    k.swizzle = (int)swizzle;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        k.es[i] = elem_strides[i];
        if (i + 1 < rank) k.strides[i] = strides_bytes[i];
    }
    std::lock_guard<std::mutex> lock(g_map_mu);
    ++g_map_clock;
    for (int i = 0; i < g_nmaps; ++i)
        if (memcmp(&g_maps[i].key, &k, sizeof k) == 0) {
            g_maps[i].used = g_map_clock;
            *map = g_maps[i].map;
            return 0;
        }
    EncodeTiledFn fn = get_encode();
    if (!fn) return 1;
    CUresult r = fn(map, dtype, (cuuint32_t)rank, addr, dims, strides_bytes, box, elem_strides,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return 1;
    int slot = g_nmaps;
    if (g_nmaps < kMapCache) {
        ++g_nmaps;
    } else {
        slot = 0;
        for (int i = 1; i < kMapCache; ++i)
            if (g_maps[i].used < g_maps[slot].used) slot = i;
    }
    g_maps[slot].key = k;
    g_maps[slot].map = *map;
    g_maps[slot].used = g_map_clock;
    return 0;
}

// Per-device attributes, queried once.
constexpr int kMaxDevices = 64;
struct DevInfo {
    std::once_flag once;
    int sms = 0;
    bool sm103 = false;
};
static DevInfo g_dev[kMaxDevices];

static int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

static const DevInfo* dev_info() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    DevInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
            d.sms = sms;
            d.sm103 = major == 10 && minor == 3;
        }
    });
    return &d;
}

int current_sms() {
    const DevInfo* d = dev_info();
    return d && d->sms > 0 ? d->sms : 148;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, kernel, size).
struct AttrEntry {
    int dev;
    const void* fn;
    int smem;
};
static AttrEntry g_attr[256];
static int g_nattr = 0;
static std::mutex g_attr_mu;

cudaError_t set_smem_attr(const void* fn, int smem) {
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        for (int i = 0; i < g_nattr; ++i)
            if (g_attr[i].dev == dev && g_attr[i].fn == fn && g_attr[i].smem >= smem) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (g_nattr < 256) g_attr[g_nattr++] = AttrEntry{dev, fn, smem};
    return cudaSuccess;
}

// SM count of the current device, 0 if it is not an sm_103 part.
static int device_sms(bool require_sm103) {
    const DevInfo* d = dev_info();
    if (!d || d->sms <= 0) return 0;
    if (require_sm103 && !d->sm103) return 0;
    return d->sms;
}

static std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
static std::atomic<int> g_debug_stall{0};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
int debug_stall() { return g_debug_stall.load(); }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool pow2_heads(int H) { return H >= 1 && H <= 128 && (H & (H - 1)) == 0; }

// Shared shape rules of the scoring calls (heads a power of two <= 128,
// index_dim a multiple of 16: "deepseek_v41.indexer" page, queries parameter).
// Rows (b, s) and query tiles are counted in int by the kernels.
static int check_dims(int64_t B, int64_t S, int64_t Skv, int H, int D) {
    if (B < 1 || S < 1 || Skv < 0) return LIDX_ERR_SHAPE;
    if (!pow2_heads(H) || D < 16 || D % 16 != 0 || D > 128) return LIDX_ERR_SHAPE;
    if (S > (1 << 30) || Skv > (1 << 30) || B > (1 << 20)) return LIDX_ERR_SHAPE;
    if (B * S > (int64_t)INT_MAX) return LIDX_ERR_SHAPE;
    return LIDX_OK;
}

// Every argument rule of the V4 forward that needs no device.
int check_fwd(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                     int64_t Skv, int H, int D, int compress_ratio, const int32_t* ks,
                     const int32_t* ke, int topk, int act, const int32_t* topk_indices_in,
                     const float* logits_out, const int32_t* indices_out, const float* scores_out) {
    if (!q || (!k && Skv > 0) || !w || !indices_out || !scores_out) return LIDX_ERR_NULL;
    if ((ks == nullptr) != (ke == nullptr)) return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if ((!ks && compress_ratio < 1) || topk < 1 || topk > (1 << 20) || (act != 0 && act != 1))
        return LIDX_ERR_SHAPE;
    if (B * S * (int64_t)topk > ((int64_t)1 << 40)) return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || (logits_out && !aligned16(logits_out)))
        return LIDX_ERR_ALIGN;
    if (topk_indices_in && !aligned16(topk_indices_in)) return LIDX_ERR_ALIGN;
    if (!topk_indices_in && Skv > kTopkMaxKeys) return LIDX_ERR_UNSUPPORTED;  // selection span
    return LIDX_OK;
}

// The V4 forward with causal (ks == ke == NULL) or explicit per-row ranges.
static int indexer_fwd_impl(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                            int64_t Skv, int H, int D, int compress_ratio, const int32_t* ks,
                            const int32_t* ke, int topk, int act, const int32_t* topk_indices_in,
                            float* logits_out, int32_t* indices_out, float* scores_out,
                            void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_fwd(q, k, w, B, S, Skv, H, D, compress_ratio, ks, ke, topk, act, topk_indices_in,
                       logits_out, indices_out, scores_out);
    if (rc) return rc;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t nout = B * S * (int64_t)topk;
    if (Skv == 0) {
        // no keys at all: every score is -inf; given indices are copied through
        if (topk_indices_in)
            return copy_pad_launch(nout, topk_indices_in, indices_out, scores_out, st) == cudaSuccess
                       ? LIDX_OK
                       : LIDX_ERR_CUDA;
        return pad_launch(nout, indices_out, scores_out, st) == cudaSuccess ? LIDX_OK : LIDX_ERR_CUDA;
    }
    if (topk_indices_in && logits_out) {
        // logits were asked for: sweep them, then gather (masked entries are -inf)
        const int rc2 = lidx_indexer_logits(q, k, w, B, S, Skv, H, D, compress_ratio, ks, ke, 1, act,
                                            logits_out, stream);
        if (rc2) return rc2;
        if (extract_launch(logits_out, topk_indices_in, B * S, Skv, topk, scores_out, st) != cudaSuccess ||
            cudaMemcpyAsync(indices_out, topk_indices_in, sizeof(int32_t) * (size_t)nout,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return LIDX_ERR_CUDA;
        return LIDX_OK;
    }
    ScoreLaunch a;
    memset(&a, 0, sizeof a);
    a.p.B = (int)B;
    a.p.S = (int)S;
    a.p.Skv = (int)Skv;
    a.p.H = H;
    a.p.D = D;
    a.p.ratio = compress_ratio < 1 ? 1 : compress_ratio;
    a.p.ks = ks;
    a.p.ke = ke;
    a.p.act = act;
    a.p.w = w;
    a.p.logits = logits_out;
    a.p.clean = 1;
    a.p.topk = topk;
    a.p.idx_in = topk_indices_in;
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

}  // namespace lidx

using namespace lidx;

extern "C" {

int lidx_version(void) { return 0x000200; }

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
    int sms = device_sms(false);
    if (sms <= 0) sms = 256;  // no device: an upper bound
    if (B <= 0 || S <= 0 || Skv < 0 || !pow2_heads(H)) return 0;
    if (op == LIDX_OP_INDEXER_FWD) {
        if (logits_materialised || topk <= 0) return 0;
        return score_scratch_bytes(S, Skv, H, sms);
    }
    if (op == LIDX_OP_SCORES_V41 || op == LIDX_OP_TOPK_V41) {
        // one byte per (batch, query tile, 128-key tile): the visibility tile map
        if (Skv <= 0) return 0;
        const int64_t QT = score_query_tile(H), units = B * ((S + QT - 1) / QT);
        // the tile map: one byte per (batch, query tile, 128-key tile)
        const int64_t map = (units * ((Skv + 127) / 128) + 255) / 256 * 256;
        if (op == LIDX_OP_SCORES_V41) return (size_t)map;
        const int64_t ranges = (units * 8 + 255) / 256 * 256;  // each query tile's key-tile range
        if (logits_materialised) return (size_t)(map + ranges);
        return (size_t)(map + ranges + (B * S * Skv * 2 + 255) / 256 * 256);  // + the bf16 scores
    }
    if (op == LIDX_OP_INDEXER_BWD) return bwd_workspace_bytes(B, S, Skv, H, D, topk, sms);
    return 0;
}

int lidx_device_status(void* stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LIDX_ERR_CUDA;
    // one status word per translation unit with kernels; every one is read (and cleared)
    const int st[] = {status_score_v4(1), status_score_v4_short(1), status_score_v4_fused(1),
                      status_score_v41(1), status_misc(1), status_bwd(1)};
    int first = 0;
    for (int v : st) {
        if (v < 0) return LIDX_ERR_CUDA;
        if (v != 0 && first == 0) first = v;
    }
    return first;
}

uint64_t lidx_set_wait_limit_ns(uint64_t ns) {
    if (ns == 0) ns = kWaitLimitNs;
    return g_wait_limit_ns.exchange(ns);
}

int lidx_debug_stall_producer(int on) { return g_debug_stall.exchange(on ? 1 : 0); }

int lidx_indexer_fwd(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                     int64_t Skv, int H, int D, int compress_ratio, int topk, int act,
                     const int32_t* topk_indices_in, float* logits_out, int32_t* indices_out,
                     float* scores_out, void* workspace, size_t workspace_bytes, void* stream) {
    return indexer_fwd_impl(q, k, w, B, S, Skv, H, D, compress_ratio, nullptr, nullptr, topk, act,
                            topk_indices_in, logits_out, indices_out, scores_out, workspace,
                            workspace_bytes, stream);
}

int lidx_indexer_fwd_ranges(const void* q, const void* k, const float* w, int64_t B, int64_t S,
                            int64_t Skv, int H, int D, const int32_t* ks, const int32_t* ke,
                            int topk, int act, const int32_t* topk_indices_in, float* logits_out,
                            int32_t* indices_out, float* scores_out, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (!ks || !ke) return LIDX_ERR_NULL;
    return indexer_fwd_impl(q, k, w, B, S, Skv, H, D, 1, ks, ke, topk, act, topk_indices_in,
                            logits_out, indices_out, scores_out, workspace, workspace_bytes, stream);
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
    if (Skv > kTopkMaxKeys) return LIDX_ERR_UNSUPPORTED;
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

// V4.1 scoring into `scores_out` (bf16 [B,S,Skv]); the tile map goes to `tilemap`.
static int scores_v41_impl(const void* q, const void* k, const void* w, const uint8_t* allowed,
                           int64_t B, int64_t S, int64_t Skv, int H, int D, int act,
                           void* scores_out, uint8_t* tilemap, int2* urange, int sms, cudaStream_t st) {
    // one launch: visibility of each (query tile, key tile) block, the tensor-core
    // pass over the blocks with a visible pair, -inf over the rest
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
    a.p.tilemap = tilemap;
    a.p.urange = urange;
    a.q = q;
    a.k = k;
    a.stream = st;
    a.num_sms = sms;
    return score_v41_launch(a) == 0 ? LIDX_OK : LIDX_ERR_CUDA;
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
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)) return LIDX_ERR_WORKSPACE;
    return scores_v41_impl(q, k, w, allowed, B, S, Skv, H, D, act, scores_out, (uint8_t*)workspace, nullptr,
                           sms, (cudaStream_t)stream);
}

int lidx_indexer_topk_v41(const void* q, const void* k, const void* w, const uint8_t* allowed,
                          int64_t B, int64_t S, int64_t Skv, int H, int D, int act, int topk,
                          void* scores_out, int32_t* indices_out, void* topk_scores_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !w || !indices_out || !topk_scores_out || (Skv > 0 && (!k || !allowed)))
        return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if ((act != 0 && act != 1) || topk < 1 || topk > (1 << 20)) return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || ((uintptr_t)scores_out & 1u) ||
        ((uintptr_t)topk_scores_out & 1u))
        return LIDX_ERR_ALIGN;
    if (Skv > kTopkMaxKeys) return LIDX_ERR_UNSUPPORTED;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t rows = B * S;
    if (Skv == 0)
        return pad16_launch(rows * (int64_t)topk, indices_out, (uint16_t*)topk_scores_out, st) ==
                       cudaSuccess
                   ? LIDX_OK
                   : LIDX_ERR_CUDA;
    const size_t need =
        lidx_workspace_bytes(LIDX_OP_TOPK_V41, B, S, Skv, H, D, topk, scores_out != nullptr);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
        return LIDX_ERR_WORKSPACE;
    // workspace: tile map, then each query tile's key-tile range, then (unless kept
    // by the caller) the bf16 scores
    const size_t map_bytes = lidx_workspace_bytes(LIDX_OP_SCORES_V41, B, S, Skv, H, D, 0, 0);
    const int64_t QT = score_query_tile(H), units = B * ((S + QT - 1) / QT);
    int2* urange = (int2*)((uint8_t*)workspace + map_bytes);
    const size_t range_bytes = (size_t)(units * 8 + 255) / 256 * 256;
    uint16_t* scores =
        scores_out ? (uint16_t*)scores_out : (uint16_t*)((uint8_t*)workspace + map_bytes + range_bytes);
    rc = scores_v41_impl(q, k, w, allowed, B, S, Skv, H, D, act, scores, (uint8_t*)workspace, urange, sms, st);
    if (rc) return rc;
    return topk_rows_bf16_launch(scores, rows, (int)S, (int)Skv, urange, (int)QT, topk, indices_out,
                                 (uint16_t*)topk_scores_out, st) == cudaSuccess
               ? LIDX_OK
               : LIDX_ERR_CUDA;
}

// The backward with causal (ks == ke == NULL) or explicit per-row ranges.
static int indexer_bwd_impl(const void* q, const void* k, const float* w, const int32_t* idx,
                            const float* grad_scores, int64_t B, int64_t S, int64_t Skv, int H,
                            int D, int compress_ratio, const int32_t* ks, const int32_t* ke,
                            int topk, int act, int grad_dtype, void* dq, void* dk, float* dw,
                            void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !w || !idx || !grad_scores || !dq || !dw || (Skv > 0 && (!k || !dk)))
        return LIDX_ERR_NULL;
    if ((ks == nullptr) != (ke == nullptr)) return LIDX_ERR_NULL;
    int rc = check_dims(B, S, Skv, H, D);
    if (rc) return rc;
    if (topk < 1 || topk > (1 << 20) || (!ks && compress_ratio < 1) || (act != 0 && act != 1) ||
        (grad_dtype != 0 && grad_dtype != 1))
        return LIDX_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(w) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dw) || !aligned16(idx) || !aligned16(grad_scores))
        return LIDX_ERR_ALIGN;
    if (Skv > kTopkMaxKeys) return LIDX_ERR_UNSUPPORTED;
    const int sms = device_sms(true);
    if (sms <= 0) return LIDX_ERR_NO_DEVICE;
    const size_t need = bwd_workspace_bytes(B, S, Skv, H, D, topk, sms);
    if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)))
        return LIDX_ERR_WORKSPACE;
    BwdLaunch a;
    memset(&a, 0, sizeof a);
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
    a.ratio = compress_ratio < 1 ? 1 : compress_ratio;
    a.ks = ks;
    a.ke = ke;
    a.topk = topk;
    a.act = act;
    a.grad_dtype = grad_dtype;
    a.dq = dq;
    a.dk = dk;
    a.dw = dw;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.stream = (cudaStream_t)stream;
    a.num_sms = sms;
    return bwd_launch(a) == cudaSuccess ? LIDX_OK : LIDX_ERR_CUDA;
}

int lidx_indexer_bwd(const void* q, const void* k, const float* w, const int32_t* idx,
                     const float* grad_scores, int64_t B, int64_t S, int64_t Skv, int H, int D,
                     int compress_ratio, int topk, int act, int grad_dtype, void* dq, void* dk,
                     float* dw, void* workspace, size_t workspace_bytes, void* stream) {
    return indexer_bwd_impl(q, k, w, idx, grad_scores, B, S, Skv, H, D, compress_ratio, nullptr,
                            nullptr, topk, act, grad_dtype, dq, dk, dw, workspace, workspace_bytes,
                            stream);
}

int lidx_indexer_bwd_ranges(const void* q, const void* k, const float* w, const int32_t* idx,
                            const float* grad_scores, int64_t B, int64_t S, int64_t Skv, int H,
                            int D, const int32_t* ks, const int32_t* ke, int topk, int act,
                            int grad_dtype, void* dq, void* dk, float* dw, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (!ks || !ke) return LIDX_ERR_NULL;
    return indexer_bwd_impl(q, k, w, idx, grad_scores, B, S, Skv, H, D, 1, ks, ke, topk, act,
                            grad_dtype, dq, dk, dw, workspace, workspace_bytes, stream);
}

}  // extern "C"
