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
//   1. The row's visible scores are staged in shared memory (16-byte loads,
//      all in flight at once), taking their min and max on the way.
//   2. NB buckets linear in (max - v): bucket(v) = floor((max - v) * NB/(max-min)),
//      clamped.  IEEE subtraction and multiplication are monotone, so a lower
//      bucket always holds strictly larger scores than a higher one.
//   3. Histogram + exclusive scan give each bucket's first output position;
//      the bucket holding the topk-th element is the threshold bucket.
//   4. Members of buckets up to the threshold are scattered, grouped by
//      bucket, into shared memory.
//   5. Each candidate's position is its bucket's start plus its rank among the
//      bucket's members under (score desc, index asc); positions < topk are
//      recorded in shared memory and written out coalesced.  Many exactly equal
//      scores make a bucket large and that step quadratic in its size.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace lidx {

constexpr int kTopkBuckets = 2048;
constexpr int kTopkCandMax = 4096;  // visible keys per row the selection supports

// Histogram index of bucket b: one pad word per 32 buckets, so that lanes
// reading runs of consecutive buckets hit distinct banks.
__device__ __forceinline__ int hidx(int b) { return b + (b >> 5); }
constexpr int kTopkHist = kTopkBuckets + kTopkBuckets / 32 + 1;

struct TopkSmem {
    float row[kTopkCandMax];          // the row's visible scores, staged once
    int start[kTopkHist];             // bucket offsets (padded); after the scatter, bucket ends
    uint16_t cand[kTopkCandMax];      // candidate keys (offsets into row), grouped by bucket
    uint16_t perm[kTopkCandMax];      // key at each output position
    float red_max[32];
    float red_min[32];
    int wsum[32];
    int bstar;
};

__device__ __forceinline__ int topk_bucket(float v, float vmax, float scale) {
    float x = __fmul_rn(__fsub_rn(vmax, v), scale);
    int b = (int)x;  // x >= 0 (saturating conversion for huge x)
    return b < kTopkBuckets ? b : kTopkBuckets - 1;
}

// Selects the top `topk` of row[lo..hi) (row is global, L2-resident) into
// out_idx/out_sc.  All NT threads of the group must call it with identical
// scalar arguments; hi - lo must not exceed kTopkCandMax.
template <int NT>
__device__ void row_topk(const float* row, int lo, int hi, int topk, int32_t* out_idx,
                         float* out_sc, TopkSmem& sm, int tid, int bar_id) {
    static_assert(NT % 32 == 0 && NT <= 1024, "group size");
    constexpr int NW = NT / 32;
    constexpr int UNR = 8;  // loads in flight per thread while staging
    const int lane = tid & 31, wid = tid >> 5;
    const int n = hi > lo ? hi - lo : 0;
    const int sel = n < topk ? n : topk;
    const float ninf = __int_as_float(0xff800000);

    if (n > 0) {
        // 1. stage the row in shared memory; min / max on the way
        float vmax = ninf, vmin = __int_as_float(0x7f800000);
        int done = 0;
        if ((((uintptr_t)(row + lo)) & 15) == 0) {
            // aligned row: 16-byte loads, all of a thread's loads in flight at once
            const int n4 = n / 4;
            const float4* r4 = reinterpret_cast<const float4*>(row + lo);
            for (int base = 0; base < n4; base += NT * UNR) {
                float4 v[UNR];
#pragma unroll
                for (int k = 0; k < UNR; ++k) {
                    const int j = base + k * NT + tid;
                    v[k] = j < n4 ? r4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < UNR; ++k) {
                    const int j = base + k * NT + tid;
                    if (j < n4) {
                        reinterpret_cast<float4*>(sm.row)[j] = v[k];
                        vmax = fmaxf(fmaxf(vmax, fmaxf(v[k].x, v[k].y)), fmaxf(v[k].z, v[k].w));
                        vmin = fminf(fminf(vmin, fminf(v[k].x, v[k].y)), fminf(v[k].z, v[k].w));
                    }
                }
            }
            done = n4 * 4;
        }
        for (int base = done; base < n; base += NT * UNR) {
            float v[UNR];
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int j = base + k * NT + tid;
                v[k] = j < n ? row[lo + j] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int j = base + k * NT + tid;
                if (j < n) {
                    sm.row[j] = v[k];
                    vmax = fmaxf(vmax, v[k]);
                    vmin = fminf(vmin, v[k]);
                }
            }
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
        for (int i = tid; i < kTopkHist; i += NT) sm.start[i] = 0;
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
            for (int j = tid; j < sel; j += NT) sm.perm[j] = (uint16_t)j;
        } else {
            float scale = (float)kTopkBuckets / __fsub_rn(vmax, vmin);
            if (!(scale < __int_as_float(0x7f800000))) scale = 0.f;  // overflowed range
            // 2. histogram
#pragma unroll 4
            for (int j = tid; j < n; j += NT)
                atomicAdd(&sm.start[hidx(topk_bucket(sm.row[j], vmax, scale))], 1);
            named_bar_sync(bar_id, NT);
            // 3. exclusive scan: thread tid owns buckets [tid*PER, tid*PER + PER)
            constexpr int PER = kTopkBuckets / NT;
            static_assert(kTopkBuckets % NT == 0 && PER >= 1, "bucket split");
            int cnt[PER];
            int local = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                cnt[i] = sm.start[hidx(tid * PER + i)];
                local += cnt[i];
            }
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sm.wsum[wid] = incl;
            named_bar_sync(bar_id, NT);
            int base = incl - local;
#pragma unroll
            for (int i = 0; i < NW; ++i) base += i < wid ? sm.wsum[i] : 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int b = tid * PER + i;
                sm.start[hidx(b)] = base;
                if (base < sel && base + cnt[i] >= sel) sm.bstar = b;
                base += cnt[i];
            }
            named_bar_sync(bar_id, NT);
            const int bstar = sm.bstar;
            // 4. scatter the candidates, grouped by bucket; start[b] becomes
            //    the end of bucket b (== start of b+1) for every b <= bstar
#pragma unroll 4
            for (int j = tid; j < n; j += NT) {
                const int b = topk_bucket(sm.row[j], vmax, scale);
                if (b <= bstar) sm.cand[atomicAdd(&sm.start[hidx(b)], 1)] = (uint16_t)j;
            }
            named_bar_sync(bar_id, NT);
            // 5. rank each candidate inside its bucket [end(b-1), end(b));
            //    record the key at its output position
            const int ncand = sm.start[hidx(bstar)];
            for (int pidx = tid; pidx < ncand; pidx += NT) {
                const int j = sm.cand[pidx];
                const float v = sm.row[j];
                const int b = topk_bucket(v, vmax, scale);
                const int s0 = b == 0 ? 0 : sm.start[hidx(b - 1)], e0 = sm.start[hidx(b)];
                int rank = 0;
                for (int qq = s0; qq < e0; qq += 4) {
                    int jq[4];
                    float vq[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) jq[u] = qq + u < e0 ? sm.cand[qq + u] : j;
#pragma unroll
                    for (int u = 0; u < 4; ++u) vq[u] = sm.row[jq[u]];
#pragma unroll
                    for (int u = 0; u < 4; ++u) rank += (vq[u] > v) || (vq[u] == v && jq[u] < j);
                }
                const int pos = s0 + rank;
                if (pos < sel) sm.perm[pos] = (uint16_t)j;
            }
        }
        named_bar_sync(bar_id, NT);
        // 6. coalesced output
        for (int p = tid; p < sel; p += NT) {
            const int j = sm.perm[p];
            out_idx[p] = lo + j;
            out_sc[p] = sm.row[j];
        }
    }
    for (int j = sel + tid; j < topk; j += NT) {
        out_idx[j] = -1;
        out_sc[j] = ninf;
    }
    named_bar_sync(bar_id, NT);  // shared scratch is free for the next row
}

}  // namespace lidx
