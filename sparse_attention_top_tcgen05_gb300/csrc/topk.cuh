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
//   1. A pass over the row (16-byte loads from L2, all of a thread's loads in
//      flight at once) takes the min and max of its visible scores.  The row
//      is not staged in shared memory: the histogram and scatter passes read
//      it again from L2, which leaves room for a third concurrent row.
//   2. NB buckets linear in (max - v): bucket(v) = floor((max - v) * NB/(max-min)),
//      clamped.  IEEE subtraction and multiplication are monotone, so a lower
//      bucket always holds strictly larger scores than a higher one.
//   3. Histogram + exclusive scan give each bucket's first output position;
//      the bucket holding the topk-th element is the threshold bucket.
//   4. Members of buckets up to the threshold are scattered, grouped by
//      bucket, into shared memory as (score, key) pairs, so that the next step
//      reads its comparands from consecutive words instead of gathering them
//      from the row (bank conflicts).
//   5. Each candidate's position is its bucket's start plus its rank among the
//      bucket's members under (score desc, index asc); positions < topk are
//      written straight to the output.  Many exactly equal scores make a
//      bucket large and that step quadratic in its size.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace lidx {

constexpr int kTopkBuckets = 1536;
constexpr int kTopkCandMax = 4096;  // visible keys per row the selection supports

// Histogram index of bucket b: one pad word per 32 buckets, so that lanes
// reading runs of consecutive buckets hit distinct banks.
__device__ __forceinline__ int hidx(int b) { return b + (b >> 5); }
constexpr int kTopkHist = kTopkBuckets + kTopkBuckets / 32 + 1;

struct TopkSmem {
    float cval[kTopkCandMax];         // candidate scores, grouped by bucket
    int start[kTopkHist];             // bucket offsets (padded); after the scatter, bucket ends
    uint16_t cidx[kTopkCandMax];      // candidate keys (offsets from lo), same order as cval
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

// Calls f(j, v) for every visible score v = r[j], j < n, of this thread's
// share: 16-byte loads, UNR of them in flight, when r is 16-byte aligned.
template <int NT, int UNR, class F>
__device__ __forceinline__ void row_pass(const float* r, int n, int tid, F&& f) {
    int done = 0;
    if ((((uintptr_t)r) & 15) == 0) {
        const int n4 = n / 4;
        const float4* r4 = reinterpret_cast<const float4*>(r);
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
                    f(4 * j, v[k].x);
                    f(4 * j + 1, v[k].y);
                    f(4 * j + 2, v[k].z);
                    f(4 * j + 3, v[k].w);
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
            v[k] = j < n ? r[j] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int j = base + k * NT + tid;
            if (j < n) f(j, v[k]);
        }
    }
}

// Selects the top `topk` of row[lo..hi) (row is global, L2-resident) into
// out_idx/out_sc.  All NT threads of the group must call it with identical
// scalar arguments; hi - lo must not exceed kTopkCandMax.
template <int NT>
__device__ void row_topk(const float* row, int lo, int hi, int topk, int32_t* out_idx,
                         float* out_sc, TopkSmem& sm, int tid, int bar_id) {
    static_assert(NT % 32 == 0 && NT <= 1024, "group size");
    constexpr int NW = NT / 32;
    constexpr int UNR = 4;  // 16-byte loads in flight per thread in each pass over the row
    const int lane = tid & 31, wid = tid >> 5;
    const int n = hi > lo ? hi - lo : 0;
    const int sel = n < topk ? n : topk;
    const float ninf = __int_as_float(0xff800000);

    if (n > 0) {
        // 1. min / max of the visible scores
        const float* r = row + lo;
        float vmax = ninf, vmin = __int_as_float(0x7f800000);
        row_pass<NT, UNR>(r, n, tid, [&](int, float v) {
            vmax = fmaxf(vmax, v);
            vmin = fminf(vmin, v);
        });
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
            for (int j = tid; j < sel; j += NT) {
                out_idx[j] = lo + j;
                out_sc[j] = r[j];
            }
        } else {
            float scale = (float)kTopkBuckets / __fsub_rn(vmax, vmin);
            if (!(scale < __int_as_float(0x7f800000))) scale = 0.f;  // overflowed range
            // 2. histogram (second pass over the row)
            row_pass<NT, UNR>(r, n, tid, [&](int, float v) {
                atomicAdd(&sm.start[hidx(topk_bucket(v, vmax, scale))], 1);
            });
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
            row_pass<NT, UNR>(r, n, tid, [&](int j, float v) {
                const int b = topk_bucket(v, vmax, scale);
                if (b <= bstar) {
                    const int pidx = atomicAdd(&sm.start[hidx(b)], 1);
                    sm.cval[pidx] = v;
                    sm.cidx[pidx] = (uint16_t)j;
                }
            });
            named_bar_sync(bar_id, NT);
            // 5. rank each candidate inside its bucket [end(b-1), end(b)) and
            //    write it at its output position
            const int ncand = sm.start[hidx(bstar)];
            for (int pidx = tid; pidx < ncand; pidx += NT) {
                const float v = sm.cval[pidx];
                const int j = sm.cidx[pidx];
                const int b = topk_bucket(v, vmax, scale);
                const int s0 = b == 0 ? 0 : sm.start[hidx(b - 1)], e0 = sm.start[hidx(b)];
                int rank = 0;
                for (int qq = s0; qq < e0; qq += 4) {
                    float vq[4];
                    int jq[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const bool in = qq + u < e0;
                        vq[u] = in ? sm.cval[qq + u] : v;
                        jq[u] = in ? (int)sm.cidx[qq + u] : j;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) rank += (vq[u] > v) || (vq[u] == v && jq[u] < j);
                }
                const int pos = s0 + rank;
                if (pos < sel) {
                    out_idx[pos] = lo + j;
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
