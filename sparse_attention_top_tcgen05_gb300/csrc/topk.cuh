// topk.cuh -- per-row top-k of scores by one group of NT threads that share a
// named barrier.  Used by the fused scoring kernel after each query tile's key
// sweep, by the standalone selection kernel over fp32 logits, and by the
// selection over V4.1 bf16 scores.
//
// Order: score descending, equal scores by ascending key index (the indexer
// pages leave the order unstated; this is torch.topk's sorted order with a
// deterministic tie rule).  Rows with fewer visible keys than topk end with
// index -1 / score -inf.  With SKIP_NINF, entries equal to -inf are not
// candidates (V4.1 scores are -inf exactly where a key is not visible).
//
// Method (exact; bounded cost for any distribution of scores):
//   1. A pass over the row (16-byte loads from L2, four in flight per thread)
//      takes the min, the max and the number of visible scores.
//   2. Work items: "emit the top `sel` of the row's scores v with
//      lo_v <= v <= hi_v at output positions base..base+sel".  The row itself
//      is the first item.  An item whose scores are all equal is emitted in
//      index order by a stable compaction.  Otherwise NB buckets map v to
//      floor((hi_v - v) * NB / (hi_v - lo_v)) (first item) or linearly by the
//      order-preserving 32-bit key of v (refined items); both maps are
//      monotone, so a lower bucket holds strictly larger scores.
//   3. Histogram + exclusive scan give each bucket's first output position; the
//      bucket holding position sel-1 is the last one needed.
//   4. The needed buckets are taken in windows of at most CAP members.  A
//      window's members are scattered into shared memory as (score, key)
//      pairs grouped by bucket.  A member of a bucket of at most kTopkSmall
//      members is ranked against its bucket mates and written straight to its
//      output position.  A larger bucket in which all but a few members hold
//      one score is ranked in place: the few pairwise, the rest by key index
//      through a bitmap of their keys and prefix popcounts.  Other large
//      buckets are refined (step 5) or sorted in place by a bitonic network
//      (one warp per bucket up to kTopkWarpSort members, else the whole group)
//      and then written out.
//   5. A single bucket with more than CAP members becomes a new item
//      over the exact value range of its members, bucketed by key; a few such
//      refinements end in buckets that fit or in all-equal items.  Histogram
//      and scatter combine the atomics of runs of one bucket (ties).
// A row of at most kTopkShort keys skips all this: one warp turns each entry
// into a 64-bit key (order key of the score, then the complement of its
// offset) and sorts the keys in registers.
#pragma once
#include <limits.h>
#include <stdint.h>

#include "ptx.cuh"

namespace lidx {

constexpr int kTopkBuckets = 1536;
constexpr int kTopkCap = 4096;       // members of one window held in shared memory
constexpr int kTopkSmall = 64;       // buckets up to this size are ranked pairwise
constexpr int kTopkWarpSort = 512;   // larger buckets up to this size: one warp sorts each
constexpr int kTopkMaxKeys = 65536;  // visible span of a row (16-bit candidate offsets)
constexpr int kTopkShort = 128;      // rows up to this span: one warp sorts the row in registers
// Pending refined items are disjoint.  Those refined because they exceed a
// window (> CAP members) number fewer than kTopkMaxKeys / CAP; those refined by
// choice (a bucket of more than kTopkWarpSort unequal members) at most
// kTopkStackOpt.
constexpr int kTopkStackOpt = 8;
constexpr int kTopkEqWords = 64;     // default bitmap: an all-equal bucket is ranked 2048 keys at a time
constexpr int kEqOnly = 1 << 20;     // flag in a large bucket's code: all its members hold one score

// Histogram index of bucket b: one pad word per 32 buckets, so that lanes
// reading runs of consecutive buckets hit distinct banks.  Slot hidx(NB)
// holds the item's member count.
__device__ __forceinline__ int hidx(int b) { return b + (b >> 5); }


struct TopkItem {
    float lo_v, hi_v;  // members: visible scores v with lo_v <= v <= hi_v
    int base;          // output position of the item's first member
    int sel;           // members to emit (the item's top `sel`)
    int mode;          // 0: buckets linear in value, 1: linear in the order-preserving key
};

// A group's scratch; CAP members of a row are held at a time (a window).  A
// smaller CAP takes less shared memory and more windows on long rows.
template <int CAP, int NB = kTopkBuckets, int EQW = kTopkEqWords>
struct TopkSmemT {
    static constexpr int kCap = CAP;
    static constexpr int kNB = NB;                       // value buckets of an item
    static constexpr int kHist = NB + NB / 32 + 2;       // padded histogram slots
    static constexpr int kEqWords = EQW;                 // bitmap words: 32*EQW keys a chunk
    // Buckets whose members all hold one score skip the off-score list.  Left
    // out of the default (fused-kernel) scratch, where the extra code measured
    // about 1 % slower on normal rows, which never take this path.
    static constexpr bool kEqOnlyPath = EQW > kTopkEqWords;
    static_assert(EQW % 32 == 0 && EQW >= kTopkSmall && EQW <= 256, "bitmap words");
    static constexpr int kStack = kTopkMaxKeys / CAP + kTopkStackOpt;
    static constexpr int kMed = CAP / (kTopkSmall + 1) + 1;
    float cval[CAP];              // window members, grouped by bucket
    int start[kHist];             // bucket offsets (padded); after the scatter, bucket ends
    uint16_t cidx[CAP];           // window members' keys (offsets from lo), same order as cval
    TopkItem stack[kStack];
    int med[kMed + 1];            // buckets of the window to sort (-1 - b: one dominant score)
    uint32_t eqbm[EQW];           // members of an all-equal bucket, one bit per key of a chunk
    int eqpre[EQW];               // set bits before each word of eqbm (within its warp's 32)
    float red_max[8];
    float red_min[8];
    int wsum[8];
    int bstar, nitems, nmed, whi, wbase, nbig, neq;
};
using TopkSmem = TopkSmemT<kTopkCap>;

// ------------------------------------------------------------- element types
template <class T>
__device__ __forceinline__ float topk_to_f(T v);
template <>
__device__ __forceinline__ float topk_to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float topk_to_f<uint16_t>(uint16_t v) {
    return __uint_as_float((uint32_t)v << 16);  // bf16 -> fp32 is exact
}
template <class T>
__device__ __forceinline__ T topk_from_f(float v);
template <>
__device__ __forceinline__ float topk_from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ uint16_t topk_from_f<uint16_t>(float v) {
    return (uint16_t)(__float_as_uint(v) >> 16);  // v came from a bf16: exact
}

// Order-preserving key: a larger score has a larger key; -0 and +0 share one.
__device__ __forceinline__ uint32_t topk_okey(float v) {
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// (v, j) comes before (w, k) in the output order
__device__ __forceinline__ bool topk_before(float v, int j, float w, int k) {
    return v > w || (v == w && j < k);
}

template <int NB>
struct TopkMap {
    int mode;
    float hi_v, scale;  // mode 0
    uint32_t khi;       // mode 1
    uint64_t mul;
    __device__ __forceinline__ int operator()(float v) const {
        if (mode == 0) {
            const float x = __fmul_rn(__fsub_rn(hi_v, v), scale);
            const int b = (int)x;  // x >= 0; the conversion saturates
            return b < NB ? b : NB - 1;
        }
        const uint64_t d = (uint64_t)(khi - topk_okey(v));
        return (int)((d * mul) >> 32);  // d < range, mul <= NB*2^32/range: < NB
    }
};

template <int NB>
__device__ __forceinline__ TopkMap<NB> topk_map(const TopkItem& it) {
    TopkMap<NB> m;
    m.mode = it.mode;
    m.hi_v = it.hi_v;
    float scale = (float)NB / __fsub_rn(it.hi_v, it.lo_v);
    if (!(scale < __int_as_float(0x7f800000))) scale = 0.f;  // range overflowed or underflowed
    m.scale = scale;
    m.khi = topk_okey(it.hi_v);
    const uint64_t range = (uint64_t)(m.khi - topk_okey(it.lo_v)) + 1;
    m.mul = (((uint64_t)NB) << 32) / range;
    return m;
}

// Calls f(j, v) for every entry v = r[j], j < n, of this thread's share:
// 16-byte loads, UNR of them in flight; a misaligned head and the tail are
// read one element at a time.
template <int NT, int UNR, class T, class F>
__device__ __forceinline__ void row_pass(const T* r, int n, int tid, F&& f) {
    constexpr int E = 16 / (int)sizeof(T);
    int head = (int)(((16u - ((uint32_t)(uintptr_t)r & 15u)) & 15u) / sizeof(T));
    if (head > n) head = n;
    for (int j = tid; j < head; j += NT) f(j, topk_to_f<T>(r[j]));
    const int nb = (n - head) / E;
    const uint4* r4 = reinterpret_cast<const uint4*>(r + head);
    for (int base = 0; base < nb; base += NT * UNR) {
        uint4 v[UNR];
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int j = base + k * NT + tid;
            v[k] = j < nb ? r4[j] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int j = base + k * NT + tid;
            if (j < nb) {
                const T* e = reinterpret_cast<const T*>(&v[k]);
#pragma unroll
                for (int u = 0; u < E; ++u) f(head + E * j + u, topk_to_f<T>(e[u]));
            }
        }
    }
    for (int j = head + nb * E + tid; j < n; j += NT) f(j, topk_to_f<T>(r[j]));
}

// As row_pass, but every lane of a warp calls f(j, v, valid) the same number
// of times (invalid slots included), so f may use full-warp primitives.
template <int NT, int UNR, class T, class F>
__device__ __forceinline__ void row_pass_uniform(const T* r, int n, int tid, F&& f) {
    constexpr int E = 16 / (int)sizeof(T);
    int head = (int)(((16u - ((uint32_t)(uintptr_t)r & 15u)) & 15u) / sizeof(T));
    if (head > n) head = n;
    for (int j0 = 0; j0 < head; j0 += NT) {
        const int j = j0 + tid;
        const bool ok = j < head;
        f(j, ok ? topk_to_f<T>(r[j]) : 0.f, ok);
    }
    const int nb = (n - head) / E;
    const uint4* r4 = reinterpret_cast<const uint4*>(r + head);
    for (int base = 0; base < nb; base += NT * UNR) {
        uint4 v[UNR];
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int j = base + k * NT + tid;
            v[k] = j < nb ? r4[j] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int j = base + k * NT + tid;
            const T* e = reinterpret_cast<const T*>(&v[k]);
#pragma unroll
            for (int u = 0; u < E; ++u) f(head + E * j + u, topk_to_f<T>(e[u]), j < nb);
        }
    }
    for (int j0 = head + nb * E; j0 < n; j0 += NT) {
        const int j = j0 + tid;
        const bool ok = j < n;
        f(j, ok ? topk_to_f<T>(r[j]) : 0.f, ok);
    }
}

// Group-wide min/max/sum; all NT threads call with their partial values.
template <int NT, class SM>
__device__ __forceinline__ void group_minmax_count(float& vmin, float& vmax, int& cnt, SM& sm,
                                                   int tid, int bar_id) {
    constexpr int NW = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    // the slots' earlier readers (a scan or reduction) are behind a barrier already
    if (lane == 0) {
        sm.red_max[wid] = vmax;
        sm.red_min[wid] = vmin;
        sm.wsum[wid] = cnt;
    }
    named_bar_sync(bar_id, NT);
    vmax = sm.red_max[0];
    vmin = sm.red_min[0];
    cnt = sm.wsum[0];
#pragma unroll
    for (int i = 1; i < NW; ++i) {
        vmax = fmaxf(vmax, sm.red_max[i]);
        vmin = fminf(vmin, sm.red_min[i]);
        cnt += sm.wsum[i];
    }
}

// Bitonic sort of s[0..c) (descending in topk_before order) by T threads of a
// warp (GROUP = false) or of the group (GROUP = true).  Every compare-exchange
// puts the earlier element at the lower position, so entries at c and beyond
// act as trailing sentinels that never move and need no storage.
template <int T, bool GROUP>
__device__ __forceinline__ void bitonic_desc(float* sv, uint16_t* sj, int c, int t, int bar_id) {
    int P = 1;
    while (P < c) P <<= 1;
    auto sync = [&]() {
        if constexpr (GROUP)
            named_bar_sync(bar_id, T);
        else
            __syncwarp();
    };
    auto cmpx = [&](int a, int b) {
        if (b >= c) return;
        const float va = sv[a], vb = sv[b];
        const int ja = sj[a], jb = sj[b];
        if (topk_before(vb, jb, va, ja)) {
            sv[a] = vb;
            sv[b] = va;
            sj[a] = (uint16_t)jb;
            sj[b] = (uint16_t)ja;
        }
    };
    for (int k = 2; k <= P; k <<= 1) {
        const int hk = k >> 1;
        for (int p = t; p < P / 2; p += T) {  // flip: mirror pairs of each k-block
            const int blk = p / hk, off = p % hk;
            cmpx(blk * k + off, blk * k + k - 1 - off);
        }
        sync();
        for (int j = hk >> 1; j > 0; j >>= 1) {
            for (int p = t; p < P / 2; p += T) {
                const int a = (p / j) * 2 * j + p % j;
                cmpx(a, a + j);
            }
            sync();
        }
    }
}

// Emits, in index order, the first `sel` members of an all-equal item
// (stable compaction with warp ballots; one barrier pair per NT entries).
template <int NT, class T, class SM>
__device__ void topk_emit_equal(const T* r, int n, int lo, const TopkItem& it, int32_t* out_idx,
                                T* out_sc, SM& sm, int tid, int bar_id) {
    constexpr int NW = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    int done = 0;  // members emitted before this round (uniform)
    for (int base = 0; base < n && done < it.sel; base += NT) {
        const int j = base + tid;
        bool m = false;
        float v = 0.f;
        if (j < n) {
            v = topk_to_f<T>(r[j]);
            m = v >= it.lo_v && v <= it.hi_v;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, m);
        named_bar_sync(bar_id, NT);  // previous round's wsum reads are done
        if (lane == 0) sm.wsum[wid] = __popc(bal);
        named_bar_sync(bar_id, NT);
        int before = done, total = done;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const int c = sm.wsum[i];
            before += i < wid ? c : 0;
            total += c;
        }
        if (m) {
            const int pos = before + __popc(bal & ((1u << lane) - 1u));
            if (pos < it.sel) {
                out_idx[it.base + pos] = lo + j;
                out_sc[it.base + pos] = topk_from_f<T>(v);
            }
        }
        done = total;
    }
}

// One work item of row_topk (see the method above).  All NT threads call it
// with the same item; it may push refined items onto sm.stack (thread 0).
// `cleared`: the histogram is already zero and visible to the group.
template <int NT, class T, class SM>
__device__ void topk_item(const T* r, int n, int lo, const TopkItem it, bool cleared,
                          int32_t* out_idx, T* out_sc, SM& sm, int tid, int bar_id) {
    constexpr int NW = NT / 32;
    constexpr int UNR = 4;  // 16-byte loads in flight per thread in each pass over the row
    const int lane = tid & 31, wid = tid >> 5;
    const float ninf = __int_as_float(0xff800000), pinf = __int_as_float(0x7f800000);
    auto member = [&](float v) { return v >= it.lo_v && v <= it.hi_v; };
    if (!(it.hi_v > it.lo_v)) {
        topk_emit_equal<NT, T>(r, n, lo, it, out_idx, out_sc, sm, tid, bar_id);
        return;
    }
    const auto bm = topk_map<SM::kNB>(it);
    // 2. histogram
    if (!cleared) {
        for (int i = tid; i < SM::kHist; i += NT) sm.start[i] = 0;
        if (tid == 0) {
            sm.bstar = SM::kNB - 1;  // set by the scan unless scores are not finite
            sm.nbig = 0;
        }
        named_bar_sync(bar_id, NT);
    }
    {
        // runs of one bucket in a thread's own sequence (ties) take one atomic
        int run_b = -1, run_c = 0;
        row_pass<NT, UNR>(r, n, tid, [&](int, float v) {
            if (!member(v)) return;
            const int b = bm(v);
            if (b == run_b) {
                ++run_c;
            } else {
                if (run_c) atomicAdd(&sm.start[hidx(run_b)], run_c);
                run_b = b;
                run_c = 1;
            }
        });
        if (run_c) atomicAdd(&sm.start[hidx(run_b)], run_c);
    }
    named_bar_sync(bar_id, NT);
    // 3. exclusive scan: thread tid owns buckets [tid*PER, tid*PER + PER)
    {
        constexpr int PER = SM::kNB / NT;
        static_assert(SM::kNB % NT == 0 && PER >= 1, "bucket split");
        int c[PER];
        int local = 0, big = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            c[i] = sm.start[hidx(tid * PER + i)];
            local += c[i];
            big += c[i] > kTopkSmall;
        }
        if (big) atomicAdd(&sm.nbig, big);
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
            if (base < it.sel && base + c[i] >= it.sel) sm.bstar = b;
            base += c[i];
        }
        if (tid == NT - 1) sm.start[hidx(SM::kNB)] = base;  // member count
    }
    named_bar_sync(bar_id, NT);
    const int bstar = sm.bstar;
    const bool any_big = sm.nbig > 0;  // some bucket is too large to rank pairwise
    // 4. windows of consecutive buckets [w_lo, whi] with at most SM::kCap members.
    // start[hidx(b)] is b's first position until b is scattered, its end after.
    int w_lo = 0;
    while (w_lo <= bstar) {
        if (tid == 0) {
            const int s_lo = sm.start[hidx(w_lo)];
            int whi;
            if (sm.start[hidx(bstar + 1)] - s_lo <= SM::kCap) {
                whi = bstar;  // the rest fits in one window
            } else if (sm.start[hidx(w_lo + 1)] - s_lo > SM::kCap) {
                whi = -1;  // one bucket too large for a window
            } else {
                int a = w_lo, b = bstar;  // largest whi in [a, b] whose window fits
                while (a < b) {
                    const int mid = (a + b + 1) >> 1;
                    if (sm.start[hidx(mid + 1)] - s_lo <= SM::kCap)
                        a = mid;
                    else
                        b = mid - 1;
                }
                whi = a;
            }
            sm.whi = whi;
            sm.wbase = s_lo;
            sm.nmed = 0;
        }
        named_bar_sync(bar_id, NT);
        const int whi = sm.whi, wbase = sm.wbase;
        if (whi < 0) {
            // refine bucket w_lo: the exact value range of its members, bucketed by key
            const int b0 = w_lo;
            float bmax = ninf, bmin = pinf;
            int bc = 0;
            row_pass<NT, UNR>(r, n, tid, [&](int, float v) {
                if (member(v) && bm(v) == b0) {
                    bmax = fmaxf(bmax, v);
                    bmin = fminf(bmin, v);
                    ++bc;
                }
            });
            group_minmax_count<NT>(bmin, bmax, bc, sm, tid, bar_id);
            if (tid == 0) {
                const int bend = sm.start[hidx(b0 + 1)];
                TopkItem ch;
                ch.lo_v = bmin;
                ch.hi_v = bmax;
                ch.base = it.base + wbase;
                const int want = it.sel - wbase;
                ch.sel = want < bc ? want : bc;
                ch.mode = 1;
                if (sm.nitems < SM::kStack) sm.stack[sm.nitems++] = ch;
                sm.start[hidx(b0)] = bend;  // as if scattered: b0 + 1 finds its start
            }
            named_bar_sync(bar_id, NT);
            w_lo = b0 + 1;
            continue;
        }
        // scatter the window's members, grouped by bucket
        if (!any_big) {
            row_pass<NT, UNR>(r, n, tid, [&](int j, float v) {
                if (!member(v)) return;
                const int b = bm(v);
                if (b >= w_lo && b <= whi) {
                    const int p = atomicAdd(&sm.start[hidx(b)], 1) - wbase;
                    sm.cval[p] = v;
                    sm.cidx[p] = (uint16_t)j;
                }
            });
        } else {
            // large buckets: lanes of a warp landing in one bucket take one atomic
            row_pass_uniform<NT, UNR>(r, n, tid, [&](int j, float v, bool ok) {
                int b = -1;
                if (ok && member(v)) {
                    b = bm(v);
                    if (b < w_lo || b > whi) b = -1;
                }
                const uint32_t peers = __match_any_sync(0xffffffffu, b);
                if (b < 0) return;
                const int leader = __ffs(peers) - 1;
                int p0 = 0;
                if (lane == leader) p0 = atomicAdd(&sm.start[hidx(b)], __popc(peers));
                p0 = __shfl_sync(peers, p0, leader);
                const int p = p0 + __popc(peers & ((1u << lane) - 1u)) - wbase;
                sm.cval[p] = v;
                sm.cidx[p] = (uint16_t)j;
            });
        }
        named_bar_sync(bar_id, NT);
        auto bbegin = [&](int b) { return b == 0 ? 0 : sm.start[hidx(b - 1)]; };
        if (any_big)  // buckets too large to rank pairwise
            for (int b = w_lo + tid; b <= whi; b += NT)
                if (sm.start[hidx(b)] - bbegin(b) > kTopkSmall) {
                    const int k = atomicAdd(&sm.nmed, 1);
                    if (k < SM::kMed) sm.med[k] = b;
                }
        // rank each member of a small bucket [begin(b), end(b)) and write it out
        const int wend = sm.start[hidx(whi)] - wbase;
        for (int p = tid; p < wend; p += NT) {
            const float v = sm.cval[p];
            const int j = sm.cidx[p];
            const int b = bm(v);
            const int s0 = bbegin(b) - wbase, e0 = sm.start[hidx(b)] - wbase;
            if (any_big && e0 - s0 > kTopkSmall) continue;
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
                for (int u = 0; u < 4; ++u) rank += topk_before(vq[u], jq[u], v, j);
            }
            const int pos = s0 + wbase + rank;
            if (pos < it.sel) {
                out_idx[it.base + pos] = lo + j;
                out_sc[it.base + pos] = topk_from_f<T>(v);
            }
        }
        if (any_big) {
            // sort the large buckets in place, then write them out
            named_bar_sync(bar_id, NT);
            const int nmed = sm.nmed < SM::kMed ? sm.nmed : SM::kMed;
            // A bucket in which all but at most kTopkSmall members hold one score
            // v0 is ranked in place (code -1 - b): members above v0 first, then
            // those equal to v0 in key order, then those below.  One of more
            // than kTopkWarpSort members without such a score is refined as an
            // item of its own over its members' exact range, while the stack has
            // room for optional items (code INT_MIN).  Others are sorted.
            for (int i = wid; i < nmed; i += NW) {
                const int b = sm.med[i];
                const int s0 = bbegin(b) - wbase, e0 = sm.start[hidx(b)] - wbase;
                const float v0 = sm.cval[s0];
                float mn = v0, mx = v0;
                int ne = 0;
                for (int p = s0 + lane; p < e0; p += 32) {
                    const float v = sm.cval[p];
                    mn = fminf(mn, v);
                    mx = fmaxf(mx, v);
                    ne += v != v0;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    ne += __shfl_xor_sync(0xffffffffu, ne, o);
                }
                if (lane == 0) {
                    if (ne <= kTopkSmall) {
                        sm.med[i] = -1 - b - ((SM::kEqOnlyPath && ne == 0) ? kEqOnly : 0);
                    } else if (e0 - s0 > kTopkWarpSort) {
                        const int slot = atomicAdd(&sm.nitems, 1);
                        if (slot < kTopkStackOpt) {
                            TopkItem ch;
                            ch.lo_v = mn;
                            ch.hi_v = mx;
                            ch.base = it.base + bbegin(b);
                            const int want = it.sel - bbegin(b);
                            ch.sel = want < e0 - s0 ? want : e0 - s0;
                            ch.mode = 1;
                            sm.stack[slot] = ch;
                            sm.med[i] = INT_MIN;
                        } else {
                            atomicSub(&sm.nitems, 1);  // no room: sorted below instead
                        }
                    }
                }
            }
            if (tid == 0) sm.neq = 0;
            named_bar_sync(bar_id, NT);
            for (int i = 0; i < nmed; ++i) {
                const int code = sm.med[i];
                if (code >= 0 || code == INT_MIN) continue;
                const bool only = SM::kEqOnlyPath && -1 - code >= kEqOnly;  // every member holds v0
                const int b = SM::kEqOnlyPath ? (-1 - code) & (kEqOnly - 1) : -1 - code;
                const int s0 = bbegin(b) - wbase, e0 = sm.start[hidx(b)] - wbase;
                const int bb = bbegin(b);  // item-local position of the bucket
                const float v0 = sm.cval[s0];
                // members off the dominant score (at most kTopkSmall): list, then rank
                int neq = 0, gt = 0;
                if (!only) {
                    for (int p = s0 + tid; p < e0; p += NT)
                        if (sm.cval[p] != v0) sm.eqpre[atomicAdd(&sm.neq, 1)] = p;
                    named_bar_sync(bar_id, NT);
                    neq = sm.neq;
                    for (int x = 0; x < neq; ++x) gt += sm.cval[sm.eqpre[x]] > v0;
                }
                if (tid < neq) {
                    const int p = sm.eqpre[tid];
                    const float v = sm.cval[p];
                    const int j = sm.cidx[p];
                    const bool above = v > v0;
                    int rank = 0;
                    for (int x = 0; x < neq; ++x) {
                        const int q = sm.eqpre[x];
                        const float vq = sm.cval[q];
                        rank += ((vq > v0) == above) && topk_before(vq, sm.cidx[q], v, j);
                    }
                    const int pos = bb + (above ? rank : gt + (e0 - s0 - neq) + rank);
                    if (pos < it.sel) {
                        out_idx[it.base + pos] = lo + j;
                        out_sc[it.base + pos] = topk_from_f<T>(v);
                    }
                }
                if (!only) named_bar_sync(bar_id, NT);  // the list is read; eqpre is reused below
                // members equal to v0: rank of key j = set bits below j in a bitmap
                constexpr int EQW = SM::kEqWords, EQK = 32 * EQW;
                static_assert(NT >= EQW, "one thread per bitmap word");
                int before = 0;  // such members in earlier chunks
                for (int c0 = 0; c0 < n; c0 += EQK) {
                    for (int x = tid; x < EQW; x += NT) sm.eqbm[x] = 0u;
                    named_bar_sync(bar_id, NT);
                    for (int p = s0 + tid; p < e0; p += NT) {
                        const int j = (int)sm.cidx[p] - c0;
                        if ((only || sm.cval[p] == v0) && j >= 0 && j < EQK)
                            atomicOr(&sm.eqbm[j >> 5], 1u << (j & 31));
                    }
                    named_bar_sync(bar_id, NT);
                    if (tid < EQW) {
                        const int cnt = __popc(sm.eqbm[tid]);
                        int incl = cnt;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const int y = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += y;
                        }
                        sm.eqpre[tid] = incl - cnt;
                        if (lane == 31) sm.wsum[wid] = incl;
                    }
                    named_bar_sync(bar_id, NT);
                    int wpre[EQW / 32];  // set bits in the words of earlier scanning warps
                    wpre[0] = 0;
#pragma unroll
                    for (int x = 1; x < EQW / 32; ++x) wpre[x] = wpre[x - 1] + sm.wsum[x - 1];
                    for (int p = s0 + tid; p < e0; p += NT) {
                        const int j = (int)sm.cidx[p] - c0;
                        if ((!only && sm.cval[p] != v0) || j < 0 || j >= EQK) continue;
                        const int wd = j >> 5;
                        int off = 0;
#pragma unroll
                        for (int x = 1; x < EQW / 32; ++x) off = (wd >> 5) == x ? wpre[x] : off;
                        const int rank = before + sm.eqpre[wd] + off +
                                         __popc(sm.eqbm[wd] & ((1u << (j & 31)) - 1u));
                        const int pos = bb + gt + rank;
                        if (pos < it.sel) {
                            out_idx[it.base + pos] = lo + sm.cidx[p];
                            out_sc[it.base + pos] = topk_from_f<T>(v0);
                        }
                    }
#pragma unroll
                    for (int x = 0; x < EQW / 32; ++x) before += sm.wsum[x];
                    if (tid == 0) sm.neq = 0;
                    named_bar_sync(bar_id, NT);
                }
            }
            for (int i = wid; i < nmed; i += NW) {
                const int b = sm.med[i];
                if (b < 0) continue;
                const int s0 = bbegin(b) - wbase, e0 = sm.start[hidx(b)] - wbase;
                if (e0 - s0 > kTopkWarpSort) continue;
                bitonic_desc<32, false>(sm.cval + s0, sm.cidx + s0, e0 - s0, lane, 0);
                for (int p = s0 + lane; p < e0; p += 32) {
                    const int pos = p + wbase;
                    if (pos < it.sel) {
                        out_idx[it.base + pos] = lo + sm.cidx[p];
                        out_sc[it.base + pos] = topk_from_f<T>(sm.cval[p]);
                    }
                }
            }
            for (int i = 0; i < nmed; ++i) {
                const int b = sm.med[i];
                if (b < 0) continue;
                const int s0 = bbegin(b) - wbase, e0 = sm.start[hidx(b)] - wbase;
                if (e0 - s0 <= kTopkWarpSort) continue;
                named_bar_sync(bar_id, NT);
                bitonic_desc<NT, true>(sm.cval + s0, sm.cidx + s0, e0 - s0, tid, bar_id);
                for (int p = s0 + tid; p < e0; p += NT) {
                    const int pos = p + wbase;
                    if (pos < it.sel) {
                        out_idx[it.base + pos] = lo + sm.cidx[p];
                        out_sc[it.base + pos] = topk_from_f<T>(sm.cval[p]);
                    }
                }
            }
        }
        named_bar_sync(bar_id, NT);  // window storage is free
        w_lo = whi + 1;
    }
}

// Bitonic sort, descending, of 32*E 64-bit keys held by one warp: element
// k*32 + lane lives in x[k] of that lane.
template <int E>
__device__ __forceinline__ void warp_bitonic_desc64(uint64_t (&x)[E], int lane) {
    constexpr int N = 32 * E;
#pragma unroll
    for (int sz = 2; sz <= N; sz <<= 1) {
#pragma unroll
        for (int d = sz >> 1; d > 0; d >>= 1) {
            if (d >= 32) {  // partner in another register of this lane
                const int kd = d / 32;
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    if (k & kd) continue;
                    const bool desc = ((k * 32 + lane) & sz) == 0;
                    const uint64_t a = x[k], b = x[k | kd];
                    const bool sw = desc ? a < b : a > b;
                    x[k] = sw ? b : a;
                    x[k | kd] = sw ? a : b;
                }
            } else {  // partner in this register of lane ^ d
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const int i = k * 32 + lane;
                    const uint64_t y = __shfl_xor_sync(0xffffffffu, x[k], d);
                    const bool keep_max = (((i & sz) == 0) == ((i & d) == 0));
                    x[k] = keep_max ? (x[k] > y ? x[k] : y) : (x[k] < y ? x[k] : y);
                }
            }
        }
    }
}

// A short row (n <= 32*E) selected by one warp: each entry becomes the key
// (order key of the value, then the complement of its offset), so that one
// descending sort gives the output order (equal values by ascending key).
// Scores are copied from the row.  With SKIP_NINF, -inf entries are not emitted.
template <int E, bool SKIP_NINF, class T>
__device__ void warp_topk_short(const T* r, int n, int lo, int topk, int32_t* out_idx, T* out_sc,
                                int lane) {
    const float ninf = __int_as_float(0xff800000);
    uint64_t x[E];
    int valid = 0;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int j = k * 32 + lane;
        x[k] = 0ull;  // padding sorts after every entry
        bool ok = false;
        if (j < n) {
            const float v = topk_to_f<T>(r[j]);
            ok = !SKIP_NINF || v > ninf;
            x[k] = ((uint64_t)topk_okey(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)j);
        }
        valid += __popc(__ballot_sync(0xffffffffu, ok));
    }
    warp_bitonic_desc64<E>(x, lane);
    const int sel = valid < topk ? valid : topk;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        const int i = k * 32 + lane;
        if (i < sel) {
            const int j = (int)(0xFFFFFFFFu - (uint32_t)x[k]);
            out_idx[i] = lo + j;
            out_sc[i] = r[j];
        }
    }
    for (int i = sel + lane; i < topk; i += 32) {
        out_idx[i] = -1;
        out_sc[i] = topk_from_f<T>(ninf);
    }
}

// Selects the top `topk` of row[lo..hi) into out_idx/out_sc.  All NT threads
// of the group must call it with identical scalar arguments, after a group
// barrier that ends any earlier use of `sm`; hi - lo must not exceed
// kTopkMaxKeys.  The row is global (L2-resident) and read several times.
template <int NT, bool SKIP_NINF, class T, class SM>
__device__ void row_topk(const T* row, int lo, int hi, int topk, int32_t* out_idx, T* out_sc,
                         SM& sm, int tid, int bar_id) {
    static_assert(NT % 32 == 0 && NT <= 256, "group size");
    const int n = hi > lo ? hi - lo : 0;
    const float ninf = __int_as_float(0xff800000), pinf = __int_as_float(0x7f800000);
    const T* r = row + lo;
    if (n <= kTopkShort) {  // one warp sorts the row in registers
        if (tid < 32) {
            if (n <= 32)
                warp_topk_short<1, SKIP_NINF, T>(r, n, lo, topk, out_idx, out_sc, tid);
            else if (n <= 64)
                warp_topk_short<2, SKIP_NINF, T>(r, n, lo, topk, out_idx, out_sc, tid);
            else
                warp_topk_short<4, SKIP_NINF, T>(r, n, lo, topk, out_idx, out_sc, tid);
        }
        named_bar_sync(bar_id, NT);  // the group moves on together
        return;
    }

    // 1. min, max and number of visible scores
    float vmax = ninf, vmin = pinf;
    int cnt = 0;
    if (n > 0)
        row_pass<NT, 4>(r, n, tid, [&](int, float v) {
            if (SKIP_NINF && !(v > ninf)) return;
            vmax = fmaxf(vmax, v);
            vmin = fminf(vmin, v);
            ++cnt;
        });
    // clear the first item's histogram under the same barrier
    for (int i = tid; i < SM::kHist; i += NT) sm.start[i] = 0;
    if (tid == 0) {
        sm.nitems = 0;
        sm.bstar = SM::kNB - 1;
        sm.nbig = 0;
    }
    group_minmax_count<NT>(vmin, vmax, cnt, sm, tid, bar_id);
    const int nvalid = SKIP_NINF ? cnt : n;
    const int sel = nvalid < topk ? nvalid : topk;

    if (sel > 0) {
        TopkItem top;
        top.lo_v = vmin;
        top.hi_v = vmax;
        top.base = 0;
        top.sel = sel;
        top.mode = 0;
        topk_item<NT, T>(r, n, lo, top, true, out_idx, out_sc, sm, tid, bar_id);
        // every push happened before a barrier inside the item
        while (sm.nitems > 0) {  // refined items (rare)
            const TopkItem it = sm.stack[sm.nitems - 1];
            named_bar_sync(bar_id, NT);  // everyone holds the item
            if (tid == 0) sm.nitems -= 1;
            topk_item<NT, T>(r, n, lo, it, false, out_idx, out_sc, sm, tid, bar_id);
            named_bar_sync(bar_id, NT);
        }
    }
    for (int j = sel + tid; j < topk; j += NT) {
        out_idx[j] = -1;
        out_sc[j] = topk_from_f<T>(ninf);
    }
    named_bar_sync(bar_id, NT);  // shared scratch is free for the next row
}

}  // namespace lidx
