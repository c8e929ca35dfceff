// topk.cuh -- per-row top-k of fp32 scores by one group of NT threads that
// share a named barrier.  Used by the fused scoring kernel after each query
// tile's key sweep, and by the standalone selection kernel.
//
// Order: score descending, equal scores by ascending key index (the indexer
// pages leave the order unstated; this is torch.topk's sorted order with a
// deterministic tie rule).  Rows with fewer visible keys than topk end with
// index -1 / score -inf.
//
// Method (value-linear bucketing, exact):
//   1. min and max of the row's visible scores.
//   2. NB buckets linear in (max - v): bucket(v) = floor((max - v) * NB/(max-min)),
//      clamped.  IEEE subtraction and multiplication are monotone, so a lower
//      bucket always holds strictly larger scores than a higher one.
//   3. Histogram + exclusive scan give each bucket's first output position;
//      the bucket holding the topk-th element is the threshold bucket.
//   4. Members of buckets up to the threshold are scattered, grouped by
//      bucket, into shared memory.
//   5. Each member's final position is its bucket's start plus its rank among
//      the bucket's members under (score desc, index asc); positions < topk
//      are written.  Buckets are small for continuous scores; many exactly
//      equal scores make a bucket large and that step quadratic in its size.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace lidx {

constexpr int kTopkBuckets = 2048;
constexpr int kTopkCandMax = 4096;  // visible keys per row the selection supports

struct TopkSmem {
    int start[kTopkBuckets + 1];
    int cursor[kTopkBuckets];
    float cand_v[kTopkCandMax];
    int cand_i[kTopkCandMax];
    float red_max[32];
    float red_min[32];
    int wsum[32];
    int bstar;
};

__device__ __forceinline__ int topk_bucket(float v, float vmax, float scale) {
    float x = __fmul_rn(__fsub_rn(vmax, v), scale);
    int b = (int)x;  // x >= 0 and finite
    return b < kTopkBuckets ? b : kTopkBuckets - 1;
}

// Selects the top `topk` of row[lo..hi) (row is global, L2-resident).
// All NT threads of the group must call it with identical scalar arguments.
template <int NT>
__device__ void row_topk(const float* row, int lo, int hi, int topk, int32_t* out_idx,
                         float* out_sc, TopkSmem& sm, int tid, int bar_id) {
    static_assert(NT % 32 == 0 && NT <= 1024, "group size");
    constexpr int NW = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    const int n = hi > lo ? hi - lo : 0;
    const int sel = n < topk ? n : topk;
    const float ninf = __int_as_float(0xff800000);

    if (n > 0) {
        // 1. min / max
        float vmax = ninf, vmin = __int_as_float(0x7f800000);
        for (int t = lo + tid; t < hi; t += NT) {
            float v = row[t];
            vmax = fmaxf(vmax, v);
            vmin = fminf(vmin, v);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
            vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
        }
        if (lane == 0) {
            sm.red_max[wid] = vmax;
            sm.red_min[wid] = vmin;
        }
        named_bar_sync(bar_id, NT);
        vmax = sm.red_max[0];
        vmin = sm.red_min[0];
#pragma unroll
        for (int i = 1; i < NW; ++i) {
            vmax = fmaxf(vmax, sm.red_max[i]);
            vmin = fminf(vmin, sm.red_min[i]);
        }

        if (!(vmax > vmin)) {
            // every visible score is equal: the first `sel` keys in index order
            for (int j = tid; j < sel; j += NT) {
                out_idx[j] = lo + j;
                out_sc[j] = row[lo + j];
            }
        } else {
            float scale = (float)kTopkBuckets / __fsub_rn(vmax, vmin);
            if (!(scale < __int_as_float(0x7f800000))) scale = 0.f;  // overflowed range
            // 2. histogram
            for (int i = tid; i <= kTopkBuckets; i += NT) sm.start[i] = 0;
            named_bar_sync(bar_id, NT);
            for (int t = lo + tid; t < hi; t += NT) atomicAdd(&sm.start[topk_bucket(row[t], vmax, scale)], 1);
            named_bar_sync(bar_id, NT);
            // 3. exclusive scan; each thread owns a run of consecutive buckets
            constexpr int PER = kTopkBuckets / NT;
            static_assert(kTopkBuckets % NT == 0, "bucket split");
            int cnt[PER];
            int local = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                cnt[i] = sm.start[tid * PER + i];
                local += cnt[i];
            }
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.wsum[wid] = incl;
            named_bar_sync(bar_id, NT);
            int base = incl - local;
            for (int i = 0; i < wid; ++i) base += sm.wsum[i];
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int b = tid * PER + i;
                sm.start[b] = base;
                sm.cursor[b] = base;
                if (base < sel && base + cnt[i] >= sel) sm.bstar = b;
                base += cnt[i];
            }
            if (tid == NT - 1) sm.start[kTopkBuckets] = base;  // == n
            named_bar_sync(bar_id, NT);
            const int bstar = sm.bstar;
            const int ncand = sm.start[bstar + 1];
            // 4. scatter the candidates, grouped by bucket
            for (int t = lo + tid; t < hi; t += NT) {
                float v = row[t];
                int b = topk_bucket(v, vmax, scale);
                if (b <= bstar) {
                    int slot = atomicAdd(&sm.cursor[b], 1);
                    sm.cand_v[slot] = v;
                    sm.cand_i[slot] = t;
                }
            }
            named_bar_sync(bar_id, NT);
            // 5. rank inside the bucket
            for (int p = tid; p < ncand; p += NT) {
                float v = sm.cand_v[p];
                int t = sm.cand_i[p];
                int b = topk_bucket(v, vmax, scale);
                int s0 = sm.start[b], e0 = sm.start[b + 1];
                int rank = 0;
                for (int qq = s0; qq < e0; ++qq) {
                    float vq = sm.cand_v[qq];
                    int iq = sm.cand_i[qq];
                    rank += (vq > v) || (vq == v && iq < t);
                }
                int pos = s0 + rank;
                if (pos < sel) {
                    out_idx[pos] = t;
                    out_sc[pos] = v;
                }
            }
        }
    }
    for (int j = sel + tid; j < topk; j += NT) {
        out_idx[j] = -1;
        out_sc[j] = ninf;
    }
    named_bar_sync(bar_id, NT);  // shared scratch is free for the next row
}

}  // namespace lidx
