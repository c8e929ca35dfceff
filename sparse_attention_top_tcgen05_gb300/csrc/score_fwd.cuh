// score_fwd.cuh -- V4 and V4.1 lightning-indexer forward on sm_103a tensor cores.
//
// Computes, for a tile of query rows against every visible compressed key,
//     logit[b,s,t] = sum_h w[s,b,h] * act(q[s,b,h,:] . k[t,b,:])
// ("tilelang_indexer" page, V4IndexerFunction: SBHD layouts; "tilelang_indexer_fwd"
// page, batched_indexer_fwd / indexer_fwd_interface / clean_logits_ /
// _make_causal_cu_seqlens), then optionally the per-row top-k; and the V4.1
// bf16-rounded scores under an explicit visibility tensor ("deepseek_v41.indexer"
// page, indexer_scores).
//
// Design (one persistent CTA per SM, warp-specialised):
//   * The contraction is oriented keys x (query, head): UMMA M = 128 keys,
//     N = 256 columns = QT queries x H heads, K = D.  Each TMEM lane is one key,
//     so the head reduction sum_h w*act(x) is a per-thread loop over columns
//     with no cross-lane traffic, and logits stores are 128 consecutive keys.
//   * warp 0 lane 0: TMA producer.  The query tile [QT*H rows, D] stays resident
//     for the whole key sweep (V4.1 keeps two); key tiles [128, D] stream through
//     a 2-stage ring.
//   * warp 1 lane 0: tcgen05.mma issuer into two 256-column fp32 accumulators
//     (512 TMEM columns), so the MMA of tile i+1 overlaps the epilogue of tile i.
//   * V4: warps 2..9, epilogue, two warps per TMEM lane quadrant (128 columns
//     each): tcgen05.ld -> act -> weighted head sum in fp32 -> mask -> store
//     (logits) or stash in one of two per-CTA L2-resident row buffers.  Warps
//     10..27 select, in three groups of six warps (topk.cuh), or one warp per row
//     when rows are short: selector g takes rows g, g+G, ... of the CTA's query
//     tiles from the row buffer the epilogue is not writing, so selection
//     overlaps the next tile's key sweep.
//   * V4.1: warps 2..17 (H <= 64) are the epilogue (bf16 rounding as the page
//     states it); the remaining warps read `allowed`, publish each query tile's
//     record of key tiles with a visible pair one unit ahead through a ring in
//     shared memory, and write -inf over the blocks with none.
//   * Key tiles with no visible pair are never loaded or multiplied.  Query
//     tiles are dealt to CTAs heaviest-first in a snake order; the next tile's
//     queries are prefetched into L2 while the current one is swept.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>
#include <stdint.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace lidx {

constexpr int kN = 256;            // UMMA N: query x head columns per tile
constexpr int kM = 128;            // UMMA M: keys per tile
constexpr int kStages = 2;         // key-tile ring depth
constexpr int kEpiWarps = 8;   // two per TMEM lane quadrant, 128 columns each
constexpr int kTopkWarps = 18;  // three selection groups of six warps
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kTopkThreads = 32 * kTopkWarps;
constexpr int kThreads = 64 + kEpiThreads + kTopkThreads;
constexpr int kEpiBar = 1;         // named barrier id of the epilogue group
constexpr int kTopkBar = 2;        // named barrier ids of the selection groups: 2, 3, 4
constexpr int kTopkGroups = 3;     // rows selected concurrently (the scratch is sized for these)
constexpr int kTopkGroupThreads = kTopkThreads / kTopkGroups;
constexpr int kTopkGroupsShort = 6;   // rows selected concurrently when Skv <= kTopkShortCap
constexpr int kTopkShortCap = 1024;   // their window: each group's scratch is a sixth of the region
constexpr int kTopkShortBuckets = 768; // and their value buckets: fewer suffice for a span that short
constexpr int kVisStages = 4;      // V4.1: ring of staged visibility blocks
constexpr int kRecSlots = 4;       // V4.1: ring of per-unit visibility records
constexpr int kFillBar = 5;        // V4.1: named barrier id of the visibility / fill warps
constexpr int kRecBitTiles = 512;  // V4.1: key tiles whose activity a record's builder keeps in bits

struct Unit {
    int b, s0, qt;
    int lo_t, hi_t;  // key tiles [lo_t, hi_t) with work
    int lo_k, hi_k;  // visible keys of the tile's union range
    uint64_t bits;   // V4.1: bit j set when key tile lo_t + j has a visible pair
};

__device__ __forceinline__ void row_range(const ScoreParams& p, int s, int& lo, int& hi) {
    if (p.ks == nullptr) {
        lo = 0;
        long long e = (long long)(s + 1) / p.ratio;
        hi = (int)(e < p.Skv ? e : p.Skv);
    } else {
        lo = p.ks[s] > 0 ? p.ks[s] : 0;
        hi = p.ke[s] < p.Skv ? p.ke[s] : p.Skv;
        if (hi < lo) hi = lo;
    }
}

template <int QT, bool V41>
__device__ __forceinline__ Unit make_unit(const ScoreParams& p, int u, const int4& rec) {
    Unit un;
    un.bits = 0;
    const int qt = p.qtiles - 1 - u / p.B;  // heaviest (latest) query tiles first
    un.b = u % p.B;
    un.qt = qt;
    un.s0 = qt * QT;
    const int s_last = min(un.s0 + QT - 1, p.S - 1);
    if constexpr (V41) {
        // the range of key tiles with visible pairs comes from the unit's record
        un.lo_t = rec.x;
        un.hi_t = rec.y;
        un.bits = (uint64_t)(uint32_t)rec.z | ((uint64_t)(uint32_t)rec.w << 32);
        un.lo_k = un.lo_t * kM;
        un.hi_k = min(un.hi_t * kM, p.Skv);
        return un;
    }
    if (p.ks == nullptr) {
        int lo, hi;
        row_range(p, s_last, lo, hi);
        un.lo_k = 0;
        un.hi_k = hi;
    } else {
        int lo = p.Skv, hi = 0;
        for (int s = un.s0; s <= s_last; ++s) {
            int a, e;
            row_range(p, s, a, e);
            if (e > a) {
                lo = min(lo, a);
                hi = max(hi, e);
            }
        }
        un.lo_k = lo;
        un.hi_k = hi;
    }
    if (un.hi_k > un.lo_k) {
        un.lo_t = un.lo_k / kM;
        un.hi_t = (un.hi_k + kM - 1) / kM;
    } else {
        un.lo_t = un.hi_t = 0;
    }
    return un;
}

template <bool V41>
__device__ __forceinline__ bool tile_active(const ScoreParams& p, const Unit& un, int kt) {
    if constexpr (V41) {
        const int j = kt - un.lo_t;
        if (j < 64) return (un.bits >> j) & 1u;
        return p.tilemap[((size_t)un.b * p.qtiles + un.qt) * p.ntk + kt] != 0;
    }
    return true;
}

// i-th unit of this CTA in snake order, or -1 when past the end
__device__ __forceinline__ int unit_of(int i, int num_units) {
    const int G = gridDim.x;
    const int base = i * G;
    if (base >= num_units) return -2;
    const int u = base + ((i & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
    return u < num_units ? u : -1;
}

// V4.1: word e of a unit's bf16 weights, laid out as the epilogue keeps them:
// heads (2e, 2e+1) of query 2e / H in one word (one weight per word at H = 1);
// zero past the sequence, for threads past the tile's words and for u < 0.
template <int H, int QT>
__device__ __forceinline__ uint32_t v41_weight_word(const ScoreParams& p, int u, int e) {
    constexpr int WPER = H >= 2 ? 2 : 1;
    if (u < 0 || e >= kN / WPER) return 0u;
    const int b = u % p.B, s = (p.qtiles - 1 - u / p.B) * QT + (WPER * e) / H, h = (WPER * e) % H;
    if (s >= p.S) return 0u;
    const uint16_t* wr = p.w16 + ((size_t)b * p.S + s) * H + h;
    if constexpr (WPER == 2) return *reinterpret_cast<const uint32_t*>(wr);  // h even: 4-byte aligned
    return (uint32_t)wr[0];
}


struct SmemLayout {
    uint32_t q_off, k_off, w_off, range_off, topk_off, bar_off, tmem_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int D) {
    SmemLayout L;
    uint32_t o = 0;
    L.q_off = o;
    o += kN * D * 2;
    L.k_off = o;
    o += kStages * kM * D * 2;
    L.w_off = o;
    o += kN * 4;
    L.range_off = o;
    o += 2 * kN * 4;
    L.topk_off = o;
    o += (uint32_t)(kTopkGroups * ((sizeof(TopkSmem) + 15) / 16 * 16));
    L.bar_off = o;
    o += 32 * 8;
    L.tmem_off = o;
    o += 16;
    L.total = o + 1024;  // slack for 1024-byte alignment of the base
    return L;
}

// (a0, a1) += (w0 * x0, w1 * x1): two fp32 fused multiply-adds in one packed
// instruction, each rounded as fmaf rounds it.
__device__ __forceinline__ void fma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
    asm("{\n\t.reg .b64 x, w, s;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 w, {%4, %5};\n\t"
        "mov.b64 s, {%0, %1};\n\tfma.rn.f32x2 s, w, x, s;\n\tmov.b64 {%0, %1}, s;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1), "f"(w0), "f"(w1));
}

// Weighted head sum sum_h w[h] * act(x[h]) of HH consecutive accumulator
// columns starting at c0 of a 32-column chunk held in registers (c0 is a
// constant once the caller's loops unroll); act is ReLU when RELU.  Four
// independent fp32 chains, two per packed instruction, weights from shared
// memory four at a time.
template <int HH, bool RELU>
__device__ __forceinline__ float head_sum_at(const uint32_t (&r)[32], int c0, const float* w) {
    auto act = [](float x) { return RELU ? fmaxf(x, 0.f) : x; };
    if constexpr (HH >= 4) {
        const float4* w4 = reinterpret_cast<const float4*>(w);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int h = 0; h < HH; h += 4) {
            const float4 wv = w4[h / 4];
            fma2(a0, a1, wv.x, wv.y, act(__uint_as_float(r[c0 + h])), act(__uint_as_float(r[c0 + h + 1])));
            fma2(a2, a3, wv.z, wv.w, act(__uint_as_float(r[c0 + h + 2])), act(__uint_as_float(r[c0 + h + 3])));
        }
        return (a0 + a1) + (a2 + a3);
    } else {
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < HH; ++h) acc = fmaf(w[h], act(__uint_as_float(r[c0 + h])), acc);
        return acc;
    }
}

// (bf16(hi) << 16) | bf16(lo), round to nearest even; RELU: negative results
// become +0 (the same as ReLU of the rounded values, up to the sign of zero,
// which a sum that starts from +0 does not see)
template <bool RELU>
__device__ __forceinline__ uint32_t cvt_bf16x2(float hi, float lo) {
    uint32_t r;
    if constexpr (RELU)
        asm("cvt.rn.relu.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// s0 += float(low half of z2), s1 += float(high half), each one fp32 add
// (the widening of a bf16 value to fp32 is exact)
__device__ __forceinline__ void add_bf16x2_f32(uint32_t z2, float& s0, float& s1) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(z2));
}
__device__ __forceinline__ float bf16_round_f(float x) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r << 16);
}

// V4.1 head reduction of one query ("deepseek_v41.indexer" page, module
// docstring): y = bf16(x); z = bf16(act(y) * w); fp32 sum of z over heads.
// wp holds the query's bf16 weights as pairs (low half = even head); for H = 1
// one weight per word.  The product of two bf16 values is exact, so rounding it
// once to bf16 is the stated rounding of the weighted head score.
template <int H, bool RELU, int NR>
__device__ __forceinline__ float head_sum_v41(const uint32_t (&r)[NR], int c0, const uint32_t* wp) {
    if constexpr (H >= 2) {
        constexpr int WV = H >= 8 ? 4 : H / 2;  // weight words per shared-memory load
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < H; h += 2 * WV) {
            uint32_t wv[WV];
            if constexpr (WV == 4) {
                const uint4 t = *reinterpret_cast<const uint4*>(wp + h / 2);
                wv[0] = t.x, wv[1] = t.y, wv[2] = t.z, wv[3] = t.w;
            } else if constexpr (WV == 2) {
                const uint2 t = *reinterpret_cast<const uint2*>(wp + h / 2);
                wv[0] = t.x, wv[1] = t.y;
            } else {
                wv[0] = wp[h / 2];
            }
#pragma unroll
            for (int j = 0; j < WV; ++j) {
                const int c = c0 + h + 2 * j;
                const uint32_t y2 = cvt_bf16x2<RELU>(__uint_as_float(r[c + 1]), __uint_as_float(r[c]));
                add_bf16x2_f32(mul_bf16x2(y2, wv[j]), s0, s1);
            }
        }
        return s0 + s1;
    } else {
        float y = bf16_round_f(__uint_as_float(r[c0]));
        if (RELU) y = fmaxf(y, 0.f);
        return bf16_round_f(y * __uint_as_float(wp[0] << 16));
    }
}

// Given-index mode ("tilelang_indexer" page, forward with topk_indices): the
// scores of the row's given keys are read back from its swept row buffer;
// a key outside the row's visible range [lo, hi) scores -inf.  Indices are
// copied through.  Ends with a group barrier like row_topk.
template <int NT>
__device__ __forceinline__ void row_gather(const float* row, int lo, int hi, const int32_t* idx,
                                           int topk, int32_t* out_idx, float* out_sc, int tid,
                                           int bar_id) {
    const float ninf = __int_as_float(0xff800000);
    for (int j = tid; j < topk; j += NT) {
        const int t = idx[j];
        out_idx[j] = t;
        out_sc[j] = (t >= lo && t < hi) ? row[t] : ninf;
    }
    named_bar_sync(bar_id, NT);
}

// V4.1: what the visibility warps gather about one unit before its record is
// written: the first and last key tile with a visible pair, and one bit per key
// tile for the first kRecBitTiles tiles.
struct RecBuild {
    int first, last;
    uint32_t bits[kRecBitTiles / 32];
};

// Configurations of the V4 kernel (template argument CFG; V4.1 takes kCfgAll):
//   kCfgAll    three selection groups; every mode of a call (materialised
//              logits, given indices, per-warp rows, either activation);
//   kCfgShort  six selection groups with windows of kTopkShortCap members, for
//              rows of at most that many keys; ReLU, fused or materialised logits,
//              no given indices or per-warp rows (7 % faster on the C4 layer than
//              with them);
//   kCfgFused  three groups, fused ReLU scoring and selection only, D = 128.
//              Leaving the other modes out of this instantiation frees registers
//              (no spills at 72 a thread) and code, and a constant D makes the
//              shared-memory layout constant: the long-context fused forward runs
//              about 9 % faster than in kCfgAll.
constexpr int kCfgAll = 0, kCfgShort = 1, kCfgFused = 2;

template <int H, bool V41, int CFG>
__global__ void __launch_bounds__(kThreads, 1)
    score_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tma, const ScoreParams p) {
    constexpr int QT = kN / H;
    constexpr bool SEL = CFG == kCfgShort, FUSED = CFG == kCfgFused;
    static_assert(!(V41 && CFG != kCfgAll), "V4.1 has one configuration");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, formed by pointer arithmetic on the shared array
    // itself so that every access through it stays a shared-memory access
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // the fused-only configuration takes D = 128: its layout is constant
    const int D = FUSED ? 128 : p.D;
    const SmemLayout L = smem_layout(D);
    uint8_t* sQ = smem + L.q_off;
    uint8_t* sK = smem + L.k_off;
    float* sW = (float*)(smem + L.w_off);
    int* sLo = (int*)(smem + L.range_off);
    int* sHi = sLo + kN;
    uint64_t* bars = (uint64_t*)(smem + L.bar_off);
    // V4.1 keeps two query tiles: the second lives in the selection scratch, which
    // V4.1 does not use, so that the next unit's queries load during this unit's
    // key sweep.  V4 keeps one.
    constexpr int NQB = V41 ? 2 : 1;
    static_assert(2 + 2 * kStages + 8 <= 14, "second query barriers overlap the ring barriers");
    // V4.1 spreads the epilogue over 16 warps of 64 accumulator columns when a
    // query's heads fit in 64 columns (the selection warps have no work there)
    constexpr int EW = (V41 && H <= 64) ? 16 : kEpiWarps;
    constexpr int EWT = 32 * EW;
    static_assert(2 + EW <= kThreads / 32, "epilogue warps exceed the block");
    // V4.1 (QT <= 32): the visibility flags of each computed block, QT rows of
    // 128 bytes, come by TMA into a ring after the second query tile
    constexpr bool VIS_RING = V41 && QT <= 32;
    // then each epilogue warp's own copy of its weights (up to 64 words a warp),
    // the record ring, the record builder's state (two) and an abort flag
    static_assert(kTopkGroups * ((sizeof(TopkSmem) + 15) / 16 * 16) >=
                      (size_t)kN * 128 * 2 + kVisStages * 32 * kM + 16 * 64 * 4 + kRecSlots * 16 +
                          2 * sizeof(RecBuild) + 16,
                  "second query tile, visibility ring, weights and records exceed the scratch");
    const bool vis_tma = VIS_RING && p.vis_tma;
    uint8_t* const sQ1 = smem + L.topk_off;  // second query tile (V4.1 only)
    uint8_t* const sVis = sQ1 + kN * D * 2;
    uint32_t* const sWw = reinterpret_cast<uint32_t*>(sVis + kVisStages * 32 * kM);  // [EW][64]
    int4* const sRec = reinterpret_cast<int4*>(sWw + 16 * 64);                        // [kRecSlots]
    RecBuild* const sBuild = reinterpret_cast<RecBuild*>(sRec + kRecSlots);           // [2]
    int* const sAbort = reinterpret_cast<int*>(sBuild + 2);
    uint64_t* vis_full = bars + 16;   // [kVisStages]
    uint64_t* vis_empty = bars + 20;  // [kVisStages]
    uint64_t* rec_full = bars + 24;   // [kRecSlots] record c written
    uint64_t* rec_empty = bars + 28;  // [kRecSlots] record c read by every other role
    auto sQb = [&](int qb) { return qb ? sQ1 : sQ; };
    auto q_fullv = [&](int qb) { return bars + (qb ? 14 : 0); };
    auto q_emptyv = [&](int qb) { return bars + (qb ? 15 : 1); };
    uint64_t* k_full = bars + 2;                  // [kStages]
    uint64_t* k_empty = bars + 2 + kStages;       // [kStages]
    uint64_t* acc_full = bars + 2 + 2 * kStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;           // [2]
    uint64_t* rows_full = acc_empty + 2;          // [2] epilogue -> top-k
    uint64_t* rows_empty = rows_full + 2;         // [2] top-k -> epilogue
    uint32_t* tmem_slot = (uint32_t*)(smem + L.tmem_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int swz = FUSED ? 128 : p.swz, KB = swz / 2, nkb = D / KB;
    const bool materialise = !V41 && !FUSED && p.logits != nullptr;
    const bool select = !V41 && p.topk > 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NQB; ++i) {
            mbar_init(q_fullv(i), 1);
            mbar_init(q_emptyv(i), 1);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(k_full + i, 1);
            mbar_init(k_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, EW);
            mbar_init(rows_full + i, kEpiThreads);
            mbar_init(rows_empty + i, QT);  // one arrival per selected row
        }
        if (vis_tma)
            for (int i = 0; i < kVisStages; ++i) {
                mbar_init(vis_full + i, 1);
                mbar_init(vis_empty + i, EW);
            }
        if (V41)
            for (int i = 0; i < kRecSlots; ++i) {
                mbar_init(rec_full + i, 1);
                mbar_init(rec_empty + i, 2 + EW);  // producer, MMA issuer, each epilogue warp
            }
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        if (vis_tma) tma_prefetch_desc(&tma);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // V4.1: record c of the CTA's sequence of units, copied out of its ring slot,
    // which is then released (one arrival per role, per epilogue warp)
    auto rec_take = [&](int c, int4& rec) -> bool {
        if (!mbar_wait(rec_full + c % kRecSlots, (c / kRecSlots) & 1, p.wait_ns)) return false;
        rec = sRec[c % kRecSlots];
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && !p.debug_stall) {
            int kcount = 0, qcount = 0;
            bool ok = true;
            int c = 0;  // units taken so far (V4.1 record index)
            for (int i = 0; ok; ++i) {
                const int u = unit_of(i, p.num_units);
                if (u == -2) break;
                if (u < 0) continue;
                int4 rec = make_int4(0, 0, 0, 0);
                if constexpr (V41) {
                    if (!(ok = rec_take(c, rec))) break;
                    mbar_arrive(rec_empty + c % kRecSlots);
                    ++c;
                }
                const Unit un = make_unit<QT, V41>(p, u, rec);
                if (un.hi_t <= un.lo_t) continue;
                const int qb = qcount % NQB;
                if (!(ok = mbar_wait(q_emptyv(qb), ((qcount / NQB) & 1) ^ 1, p.wait_ns))) break;
                ++qcount;
                mbar_arrive_expect_tx(q_fullv(qb), kN * D * 2);
                for (int kb = 0; kb < nkb; ++kb)
                {
                    if constexpr (V41)  // q [B,S,H,D]: dims (D, H, S, B)
                        tma_load_4d(sQb(qb) + kb * kN * swz, &tmq, q_fullv(qb), kb * KB, 0, un.s0, un.b);
                    else  // q [S,B,H,D]: dims (D, H, B, S)
                        tma_load_4d(sQb(qb) + kb * kN * swz, &tmq, q_fullv(qb), kb * KB, 0, un.b, un.s0);
                }
                // warm L2 with the next query tile of this CTA
                const int un2 = unit_of(i + 1, p.num_units);
                if (un2 >= 0) {
                    const int qt2 = p.qtiles - 1 - un2 / p.B;
                    for (int kb = 0; kb < nkb; ++kb)
                    {
                        if constexpr (V41)
                            tma_prefetch_l2_4d(&tmq, kb * KB, 0, qt2 * QT, un2 % p.B);
                        else
                            tma_prefetch_l2_4d(&tmq, kb * KB, 0, un2 % p.B, qt2 * QT);
                    }
                }
                for (int kt = un.lo_t; kt < un.hi_t; ++kt) {
                    if (!tile_active<V41>(p, un, kt)) continue;
                    const int kc = kcount++, st = kc % kStages;
                    if (!(ok = mbar_wait(k_empty + st, ((kc / kStages) & 1) ^ 1, p.wait_ns))) break;
                    uint8_t* dst = sK + st * kM * D * 2;
                    mbar_arrive_expect_tx(k_full + st, kM * D * 2);
                    for (int kb = 0; kb < nkb; ++kb) {
                        if constexpr (V41)  // k [B,Skv,D]: dims (D, Skv, B)
                            tma_load_3d(dst + kb * kM * swz, &tmk, k_full + st, kb * KB, kt * kM, un.b);
                        else  // k [Skv,B,D]: dims (D, B, Skv)
                            tma_load_3d(dst + kb * kM * swz, &tmk, k_full + st, kb * KB, un.b, kt * kM);
                    }
                    if (vis_tma) {  // allowed [B,S,Skv]: dims (Skv, S, B); zero past the ends
                        const int vs = kc % kVisStages;
                        if (!(ok = mbar_wait(vis_empty + vs, ((kc / kVisStages) & 1) ^ 1, p.wait_ns))) break;
                        mbar_arrive_expect_tx(vis_full + vs, QT * kM);
                        tma_load_3d(sVis + vs * QT * kM, &tma, vis_full + vs, kt * kM, un.s0, un.b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kM, kN);
            // Every descriptor the tile loop needs is built once per CTA, exactly as
            // the per-step formula builds it (address + offset, then masked).
            const int nk = D / 16;
            uint64_t ad[kStages][8], bd[8];
            {
                const uint32_t a0 = smem_u32(sK), stage = (uint32_t)(kM * D * 2), b0 = smem_u32(sQ);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int kb = (k * 16) / KB, koff = ((k * 16) % KB) * 2;
                    const uint32_t ao = (uint32_t)(kb * kM * swz + koff);
#pragma unroll
                    for (int j = 0; j < kStages; ++j) ad[j][k] = smem_desc_kmajor(a0 + j * stage + ao, swz);
                    bd[k] = smem_desc_kmajor(b0 + (uint32_t)(kb * kN * swz + koff), swz);
                }
            }
            int kcount = 0, tcount = 0, qcount = 0;
            bool ok = true;
            int c = 0;  // units taken so far (V4.1 record index)
            for (int i = 0; ok; ++i) {
                const int u = unit_of(i, p.num_units);
                if (u == -2) break;
                if (u < 0) continue;
                int4 rec = make_int4(0, 0, 0, 0);
                if constexpr (V41) {
                    if (!(ok = rec_take(c, rec))) break;
                    mbar_arrive(rec_empty + c % kRecSlots);
                    ++c;
                }
                const Unit un = make_unit<QT, V41>(p, u, rec);
                if (un.hi_t <= un.lo_t) continue;
                const int qb = qcount % NQB;
                if (!(ok = mbar_wait(q_fullv(qb), (qcount / NQB) & 1, p.wait_ns))) break;
                ++qcount;
                // the second query buffer's descriptors: the start-address field (address/16,
                // 14 bits) moves by the buffers' distance; shared addresses stay below 256 KB
                const uint64_t qdelta = qb ? (uint64_t)((smem_u32(sQ1) - smem_u32(sQ)) >> 4) : 0ull;
                tc_fence_after();
                for (int kt = un.lo_t; kt < un.hi_t; ++kt) {
                    if (!tile_active<V41>(p, un, kt)) continue;
                    const int st = kcount % kStages, acc = tcount & 1;
                    const uint32_t kph = (kcount / kStages) & 1, aph = ((tcount >> 1) & 1) ^ 1;
                    ++kcount;
                    ++tcount;
                    if (!(ok = mbar_wait(acc_empty + acc, aph, p.wait_ns))) break;
                    tc_fence_after();
                    if (!(ok = mbar_wait(k_full + st, kph, p.wait_ns))) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + acc * kN;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint64_t a = ad[0][k];
#pragma unroll
                        for (int j = 1; j < kStages; ++j) a = st == j ? ad[j][k] : a;
                        if (k < nk) umma_f16(d, a, bd[k] + qdelta, idesc, k > 0 ? 1u : 0u);
                    }
                    umma_commit(k_empty + st);
                    umma_commit(acc_full + acc);
                }
                if (ok) umma_commit(q_emptyv(qb));
            }
        }
    } else if (warp < 2 + EW) {
        // --------------------------------------------------------- epilogue
        const int etid = threadIdx.x - 64;
        const int quad = warp & 3;           // TMEM lane quadrant this warp may read
        const int half = (warp - 2) >> 2;    // which 128 of the 256 accumulator columns
        constexpr int QH = QT / 2;           // queries per half (H <= 128)
        const int row_t = quad * 32 + lane;  // key within the tile
        const float ninf = __int_as_float(0xff800000);
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        const int ntiles_all = (p.Skv + kM - 1) / kM;
        int tcount = 0, ucount = 0;
        bool ok = true;
        int c = 0;  // units taken so far (V4.1 record index)
        // V4.1: accumulator columns of this warp (64 or 128), its whole queries, and
        // its weight words per lane, held one unit ahead
        constexpr int CPW = 4 * kN / EW, QW = CPW / H, WPER = H >= 2 ? 2 : 1;
        constexpr int NWL = V41 ? CPW / WPER / 32 : 1;
        const bool relu = FUSED || SEL || p.act == 0;
        uint32_t wreg[NWL];
#pragma unroll
        for (int k = 0; k < NWL; ++k)
            wreg[k] = V41 ? v41_weight_word<H, QT>(p, unit_of(0, p.num_units), (half * CPW) / WPER + k * 32 + lane)
                          : 0u;
        for (int i = 0; ok; ++i) {
            const int u = unit_of(i, p.num_units);
            if (u == -2) break;
            if (u < 0) continue;
            int4 rec = make_int4(0, 0, 0, 0);
            if constexpr (V41) {
                if (!(ok = rec_take(c, rec))) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(rec_empty + c % kRecSlots);
                ++c;
            }
            const Unit un = make_unit<QT, V41>(p, u, rec);
            if constexpr (V41) {
                const int q0 = half * QW;  // this warp's first query within the tile
                // the bf16 weights of this warp's queries (two per word) into the warp's
                // own slot; they were loaded during the previous unit
                uint32_t* const sWp = sWw + (warp - 2) * 64;
                const int u1 = unit_of(i + 1, p.num_units);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < NWL; ++k) {
                    sWp[k * 32 + lane] = wreg[k];
                    wreg[k] = v41_weight_word<H, QT>(p, u1, (half * CPW) / WPER + k * 32 + lane);
                }
                __syncwarp();
                for (int kt = un.lo_t; kt < un.hi_t; ++kt) {
                    if (!tile_active<V41>(p, un, kt)) continue;  // written as -inf by the fill warps
                    const int t = kt * kM + row_t;
                    const int acc = tcount & 1, vs = tcount % kVisStages;
                    const uint32_t vph = (tcount / kVisStages) & 1;
                    // without the ring: this thread's flags, read before the wait so that
                    // their latency overlaps the tile's MMA (up to 8 queries a warp)
                    constexpr int QF = QW <= 8 ? QW : 1;
                    uint8_t vis[QF];
#pragma unroll
                    for (int j = 0; j < QF; ++j) {
                        const int s = un.s0 + q0 + j;
                        vis[j] = (!vis_tma && QW <= 8 && s < p.S && t < p.Skv)
                                     ? p.allowed[((size_t)un.b * p.S + s) * p.Skv + t]
                                     : (uint8_t)0;
                    }
                    if (!(ok = mbar_wait(acc_full + acc, (tcount >> 1) & 1, p.wait_ns))) break;
                    ++tcount;
                    tc_fence_after();
                    if (vis_tma && !(ok = mbar_wait(vis_full + vs, vph, p.wait_ns))) break;
                    const uint8_t* sv = sVis + vs * QT * kM + row_t;
                    auto store16 = [&](int ql, float v) {
                        const int s = un.s0 + ql;
                        if (s >= p.S || t >= p.Skv) return;
                        const size_t o = ((size_t)un.b * p.S + s) * p.Skv + t;
                        const bool visible = vis_tma     ? sv[ql * kM] != 0
                                             : QW <= 8 ? vis[(ql - q0) % QF] != 0
                                                       : p.allowed[o] != 0;
                        uint16_t bits = 0xFF80u;  // -inf
                        if (visible) bits = (uint16_t)(__float_as_uint(bf16_round_f(v)) >> 16);
                        p.out16[o] = bits;
                    };
                    float run = 0.f;
#pragma unroll
                    for (int c = 0; c < CPW / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(lane_addr + acc * kN + half * CPW + c * 32, r);
                        tmem_ld_wait();
                        if (c == CPW / 32 - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(acc_empty + acc);
                        }
                        const uint32_t* wp = sWp + (c * 32) / WPER;
                        if constexpr (H >= 32) {
                            run += relu ? head_sum_v41<32, true>(r, 0, wp) : head_sum_v41<32, false>(r, 0, wp);
                            if (((c + 1) * 32) % H == 0) {
                                store16(q0 + (c * 32) / H, run);
                                run = 0.f;
                            }
                        } else {
#pragma unroll
                            for (int qq = 0; qq < 32 / H; ++qq) {
                                const uint32_t* wq = wp + (qq * H) / WPER;
                                store16(q0 + c * (32 / H) + qq, relu ? head_sum_v41<H, true>(r, qq * H, wq)
                                                                     : head_sum_v41<H, false>(r, qq * H, wq));
                            }
                        }
                    }
                    if (vis_tma) {  // this warp is done with the staged flags
                        __syncwarp();
                        if (lane == 0) mbar_arrive(vis_empty + vs);
                    }
                }
                continue;
            }
            const int rb = ucount & 1;
            float* rows = nullptr;
            if (select) {
                // the top-k group must have finished the tile that last used slot rb
                // (this also keeps the row barriers at most one phase apart)
                if (!(ok = mbar_wait(rows_empty + rb, ((ucount >> 1) & 1) ^ 1, p.wait_ns))) break;
                if (!materialise)
                    rows = p.scratch + ((size_t)blockIdx.x * 2 + rb) * p.scratch_stride_cta;
            }
            named_bar_sync(kEpiBar, kEpiThreads);
            for (int e = etid; e < kN; e += kEpiThreads) {
                const int ql = e / H, h = e % H, s = un.s0 + ql;
                sW[e] = s < p.S ? p.w[((size_t)s * p.B + un.b) * H + h] : 0.f;
            }
            for (int ql = etid; ql < QT; ql += kEpiThreads) {
                const int s = un.s0 + ql;
                int lo = 0, hi = -1;  // hi < 0: no such query row
                if (s < p.S) row_range(p, s, lo, hi);
                sLo[ql] = lo;
                sHi[ql] = hi;
            }
            named_bar_sync(kEpiBar, kEpiThreads);
            const int t_begin = materialise ? 0 : un.lo_t;
            const int t_end = materialise ? ntiles_all : un.hi_t;
            for (int kt = t_begin; kt < t_end; ++kt) {
                const int t = kt * kM + row_t;
                const bool computed = kt >= un.lo_t && kt < un.hi_t;
                if (!computed) {
                    // tile outside every row's range: masked fill only
                    if (p.clean && t < p.Skv)
                        for (int j = 0; j < QH; ++j) {
                            const int ql = half * QH + j;
                            if (sHi[ql] >= 0)
                                p.logits[((size_t)un.b * p.S + un.s0 + ql) * p.Skv + t] = ninf;
                        }
                    continue;
                }
                const int acc = tcount & 1;
                if (!(ok = mbar_wait(acc_full + acc, (tcount >> 1) & 1, p.wait_ns))) break;
                ++tcount;
                tc_fence_after();
                auto store = [&](int ql, float v) {
                    const int lo = sLo[ql], hi = sHi[ql];
                    if (hi < 0) return;
                    const bool vis = t >= lo && t < hi;
                    if (materialise) {
                        if (t < p.Skv && (vis || p.clean))
                            p.logits[((size_t)un.b * p.S + un.s0 + ql) * p.Skv + t] = vis ? v : ninf;
                    } else if (rows) {
                        rows[(size_t)ql * p.Skv_pad + t] = v;
                    }
                };
                // this warp's 128 columns as 4 chunks of 32
                const float* wh = sW + half * 128;
                float run = 0.f;  // partial sum of a query spanning several chunks
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + acc * kN + half * 128 + c * 32, r);
                    tmem_ld_wait();
                    if (c == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty + acc);  // accumulator may be reused
                    }
                    if constexpr (H >= 32) {
                        run += relu ? head_sum_at<32, true>(r, 0, wh + c * 32)
                                    : head_sum_at<32, false>(r, 0, wh + c * 32);
                        if (((c + 1) * 32) % H == 0) {
                            store(half * QH + (c * 32) / H, run);
                            run = 0.f;
                        }
                    } else {
#pragma unroll
                        for (int qq = 0; qq < 32 / H; ++qq)
                            store(half * QH + c * (32 / H) + qq,
                                  relu ? head_sum_at<H, true>(r, qq * H, wh + c * 32 + qq * H)
                                       : head_sum_at<H, false>(r, qq * H, wh + c * 32 + qq * H));
                    }
                }
            }
            if (!ok) break;
            if (select) {
                // publish this tile's rows to the top-k group (release on arrive)
                mbar_arrive(rows_full + rb);
            }
            ++ucount;
        }
    } else if constexpr (V41) {
        // ------------------------------------------------- visibility and fill
        // The remaining warps read each unit's rows of `allowed` once, publish the
        // unit's record (its range of key tiles with a visible pair and their
        // activity bits) one unit ahead of its use, and write -inf over every block
        // of the unit that holds no visible pair, while the tensor-core sweep
        // computes the others: each output element is written once, by this fill
        // or by the epilogue.
        constexpr int FT = kThreads - 64 - EWT, FW = FT / 32;
        const int ftid = threadIdx.x - 64 - EWT, fw = ftid >> 5;
        const bool vec = (p.Skv % 8) == 0 && (((uintptr_t)p.out16) & 15) == 0;
        const bool vec16 = (p.Skv % 16) == 0 && (((uintptr_t)p.allowed) & 15) == 0;
        const bool vec4 = (p.Skv % 4) == 0 && (((uintptr_t)p.allowed) & 3) == 0;
        const uint4 ninf4 = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        const int ntk = p.ntk;
        // Record c (unit u): key-tile flags into the tile map and the builder's
        // state, then warp 0 of this role writes the ring slot.  False when the
        // slot did not come free in time.
        auto build_record = [&](int c, int u) -> bool {
            RecBuild& st = sBuild[c & 1];  // the other one may still be read by warp 0
            const int slot = c % kRecSlots;
            if (ftid == 0)
                *sAbort = mbar_wait(rec_empty + slot, ((c / kRecSlots) & 1) ^ 1, p.wait_ns) ? 0 : 1;
            if (ftid == 0) st.first = ntk;
            if (ftid == 1) st.last = -1;
            if (ftid >= 2 && ftid < 2 + kRecBitTiles / 32) st.bits[ftid - 2] = 0u;
            named_bar_sync(kFillBar, FT);
            if (*sAbort) return false;
            const int b = u % p.B, qt = p.qtiles - 1 - u / p.B, s0 = qt * QT;
            const int rows = min(QT, p.S - s0);
            uint8_t* const map = p.tilemap + ((size_t)b * p.qtiles + qt) * ntk;
            const uint8_t* const ubase = p.allowed + ((size_t)b * p.S + s0) * p.Skv;
            auto mark = [&](int kt, bool active) {
                map[kt] = active ? 1 : 0;
                if (active) {
                    atomicMin(&st.first, kt);
                    atomicMax(&st.last, kt);
                    if (kt < kRecBitTiles) atomicOr(&st.bits[kt >> 5], 1u << (kt & 31));
                }
            };
            if (vec16) {
                // a lane reads 16 flags of a row; 8 lanes cover a key tile, a warp 512 keys
                // two chunks of a warp in flight together
                const int nch = (ntk + 3) / 4;
                for (int ch0 = fw; ch0 < nch; ch0 += 2 * FW) {
                    uint32_t acc[2] = {0u, 0u};
                    bool in[2];
                    const uint8_t* base[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t0 = (ch0 + h * FW) * 512 + lane * 16;
                        in[h] = t0 < p.Skv;  // Skv % 16 == 0: all 16 keys inside or none
                        base[h] = ubase + (in[h] ? t0 : 0);
                    }
                    int r = 0;
                    for (; r + 4 <= rows; r += 4) {
                        uint4 v[2][4];
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                v[h][q] = in[h] ? *reinterpret_cast<const uint4*>(base[h] + (size_t)(r + q) * p.Skv)
                                                : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[h] |= v[h][q].x | v[h][q].y | v[h][q].z | v[h][q].w;
                    }
                    for (; r < rows; ++r)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 v = in[h] ? *reinterpret_cast<const uint4*>(base[h] + (size_t)r * p.Skv)
                                                  : make_uint4(0u, 0u, 0u, 0u);
                            acc[h] |= v.x | v.y | v.z | v.w;
                        }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t any = acc[h] != 0 ? 1u : 0u;
                        any |= __shfl_xor_sync(0xffffffffu, any, 1);
                        any |= __shfl_xor_sync(0xffffffffu, any, 2);
                        any |= __shfl_xor_sync(0xffffffffu, any, 4);
                        const int kt = (ch0 + h * FW) * 4 + (lane >> 3);
                        if ((lane & 7) == 0 && kt < ntk) mark(kt, any != 0);
                    }
                }
            } else {
                // a lane reads 4 flags of a row (one word when rows are 4-byte aligned)
                for (int kt = fw; kt < ntk; kt += FW) {
                    const int t0 = kt * kM + lane * 4;
                    uint32_t any = 0;
                    for (int r = 0; r < rows; ++r) {
                        const uint8_t* row = ubase + (size_t)r * p.Skv;
                        if (vec4 && t0 + 3 < p.Skv) {
                            any |= *reinterpret_cast<const uint32_t*>(row + t0);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (t0 + j < p.Skv) any |= row[t0 + j];
                        }
                    }
                    const bool active = __any_sync(0xffffffffu, any != 0);
                    if (lane == 0) mark(kt, active);
                }
            }
            named_bar_sync(kFillBar, FT);  // the unit's flags are all in
            if (fw == 0) {
                const int first = st.first, last = st.last;
                int4 r = make_int4(0, 0, 0, 0);
                if (last >= 0) {
                    auto active = [&](int kt) {
                        if (kt > last) return false;
                        if (kt < kRecBitTiles) return ((st.bits[kt >> 5] >> (kt & 31)) & 1u) != 0u;
                        return map[kt] != 0;
                    };
                    const uint32_t m0 = __ballot_sync(0xffffffffu, active(first + lane));
                    const uint32_t m1 = __ballot_sync(0xffffffffu, active(first + 32 + lane));
                    r = make_int4(first, last + 1, (int)m0, (int)m1);
                }
                if (lane == 0) {
                    sRec[slot] = r;
                    mbar_arrive(rec_full + slot);  // release: the record and the tile map row
                    if (p.urange) p.urange[(size_t)b * p.qtiles + qt] = make_int2(r.x, r.y);
                }
            }
            return true;
        };
        // the CTA's next unit from position i on (-2 past the end)
        auto next_unit = [&](int& i) {
            int u;
            do {
                u = unit_of(i++, p.num_units);
            } while (u == -1);
            return u;
        };
        // the rows of unit u into L2 ahead of its record (16-byte aligned rows only)
        auto prefetch_rows = [&](int u) {
            if (u < 0 || !vec16 || ftid != 0) return;
            const int b = u % p.B, s0 = (p.qtiles - 1 - u / p.B) * QT;
            const uint8_t* src = p.allowed + ((size_t)b * p.S + s0) * p.Skv;
            size_t left = (size_t)min(QT, p.S - s0) * p.Skv;  // contiguous rows
            for (; left > 0; src += 16384) {
                const uint32_t n = left < 16384 ? (uint32_t)left : 16384u;
                bulk_prefetch_l2(src, n);
                left -= n;
            }
        };
        int i = 0, c = 0;
        int u = next_unit(i);
        {
            int ip = i;
            prefetch_rows(next_unit(ip));
        }
        bool ok = u < 0 || build_record(0, u);
        while (ok && u >= 0) {
            const int u_next = next_unit(i);
            {
                int ip = i;
                prefetch_rows(next_unit(ip));  // the unit after next
            }
            if (u_next >= 0)
                ok = build_record(c + 1, u_next);  // one unit ahead of its use
            else
                named_bar_sync(kFillBar, FT);  // record c is visible to the whole role
            if (!ok) break;
            const Unit un = make_unit<QT, true>(p, u, sRec[c % kRecSlots]);
            const int rows = min(QT, p.S - un.s0);
            // keys [a, b) of every row of the unit; a and b multiples of 8 when vec
            auto fill = [&](int a, int b) {
                for (int r = 0; r < rows; ++r) {
                    uint16_t* o = p.out16 + ((size_t)un.b * p.S + un.s0 + r) * p.Skv;
                    if (vec)
                        for (int x = a + ftid * 8; x < b; x += FT * 8) *reinterpret_cast<uint4*>(o + x) = ninf4;
                    else
                        for (int x = a + ftid; x < b; x += FT) o[x] = 0xFF80u;
                }
            };
            // the key tiles before and after the unit's range, then the empty tiles inside it
            const int lo_k = un.lo_t * kM, hi_k = min(un.hi_t * kM, p.Skv);
            if (un.hi_t > un.lo_t) {
                fill(0, lo_k);
                fill(hi_k, p.Skv);
                for (int kt = un.lo_t + 1; kt < un.hi_t - 1; ++kt)
                    if (!tile_active<true>(p, un, kt)) fill(kt * kM, kt * kM + kM);
            } else {
                fill(0, p.Skv);
            }
            u = u_next;
            ++c;
        }
    } else {
        // ------------------------------------------------------------ top-k
        // Selector g selects rows g, g+G, g+2G, ... of this CTA's sequence of units
        // (QT rows each), so the load spreads evenly whatever QT is.  A selector is
        // a group of six warps, or, when every row spans at most kTopkShort keys, a
        // single warp (G = 18).  A selector waits for every unit's rows in turn, even
        // one holding none of its rows, so that it never tests a row-slot barrier
        // two phases behind.
        constexpr int NG = SEL ? kTopkGroupsShort : kTopkGroups;  // groups
        constexpr int GT = kTopkThreads / NG;                      // threads of a group
        using SMT = typename std::conditional<SEL, TopkSmemT<kTopkShortCap, kTopkShortBuckets>, TopkSmem>::type;
        constexpr uint32_t kGroupBytes = (sizeof(SMT) + 15) / 16 * 16;
        static_assert(NG * kGroupBytes <= kTopkGroups * ((sizeof(TopkSmem) + 15) / 16 * 16),
                      "selection groups exceed the scratch region");
        static_assert(kTopkBar + NG <= 16, "named barrier ids");
        const int ttid = threadIdx.x - 64 - kEpiThreads;
        const int grp = ttid / GT, gtid = ttid % GT;
        const bool by_warp = !FUSED && !SEL && p.warp_rows != 0;
        const int nsel = by_warp ? kTopkWarps : NG, sel_id = by_warp ? ttid / 32 : grp;
        SMT& sTg = *(SMT*)(smem + L.topk_off + grp * kGroupBytes);
        int i = 0, ucount = -1;
        Unit un{};
        bool ok = select;
        for (int r = sel_id; ok; r += nsel) {
            const int uc = r / QT, ql = r % QT;
            bool more = true;
            while (ok && ucount < uc) {
                int u;
                do {
                    u = unit_of(i++, p.num_units);
                } while (u == -1);
                if (u == -2) {
                    more = false;
                    break;
                }
                un = make_unit<QT, V41>(p, u, make_int4(0, 0, 0, 0));  // V4 only
                ++ucount;
                ok = mbar_wait(rows_full + (ucount & 1), (ucount >> 1) & 1, p.wait_ns);
            }
            if (!more || !ok) break;
            const int rb = uc & 1;
            const int s = un.s0 + ql;
            if (s < p.S) {
                int lo, hi;
                row_range(p, s, lo, hi);
                const size_t orow = ((size_t)un.b * p.S + s) * p.topk;
                const float* row = materialise
                                       ? p.logits + ((size_t)un.b * p.S + s) * p.Skv
                                       : p.scratch + ((size_t)blockIdx.x * 2 + rb) * p.scratch_stride_cta +
                                             (size_t)ql * p.Skv_pad;
                if (by_warp) {  // one warp sorts the row in registers
                    const int n = hi > lo ? hi - lo : 0;
                    if (n <= 32)
                        warp_topk_short<1, false, float>(row + lo, n, lo, p.topk, p.out_idx + orow,
                                                         p.out_sc + orow, lane);
                    else if (n <= 64)
                        warp_topk_short<2, false, float>(row + lo, n, lo, p.topk, p.out_idx + orow,
                                                         p.out_sc + orow, lane);
                    else
                        warp_topk_short<4, false, float>(row + lo, n, lo, p.topk, p.out_idx + orow,
                                                         p.out_sc + orow, lane);
                } else if (!FUSED && !SEL && p.idx_in) {
                    row_gather<GT>(row, lo, hi, p.idx_in + orow, p.topk, p.out_idx + orow,
                                                  p.out_sc + orow, gtid, kTopkBar + grp);
                } else {
                    row_topk<GT, false, float>(row, lo, hi, p.topk, p.out_idx + orow,
                                                              p.out_sc + orow, sTg, gtid,
                                                              kTopkBar + grp);  // ends with a group barrier
                }
            }
            if (by_warp) {
                __syncwarp();
                if (lane == 0) mbar_arrive(rows_empty + rb);  // this row's slot entry is free
            } else if (gtid == 0) {
                mbar_arrive(rows_empty + rb);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int H, bool V41, int CFG>
inline cudaError_t launch_h(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& ma, int smem, int grid) {
    auto kern = score_fwd_kernel<H, V41, CFG>;
    cudaError_t e = set_smem_attr((const void*)kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, (cudaStream_t)a.stream>>>(mq, mk, ma, a.p);
    return cudaGetLastError();
}

// Launches the kernel for the call's head count.  Each (V41, CFG) configuration
// is instantiated in a translation unit of its own (score_fwd_*.cu).
template <bool V41, int CFG>
inline cudaError_t launch_any(const ScoreLaunch& a, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& ma, int smem, int grid) {
    switch (a.p.H) {
        case 1: return launch_h<1, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 2: return launch_h<2, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 4: return launch_h<4, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 8: return launch_h<8, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 16: return launch_h<16, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 32: return launch_h<32, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 64: return launch_h<64, V41, CFG>(a, mq, mk, ma, smem, grid);
        case 128: return launch_h<128, V41, CFG>(a, mq, mk, ma, smem, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lidx
