// bwd.cu -- backward of the V4 indexer through the selected entries
// ("tilelang_indexer" page, V4IndexerFunction.backward(grad_scores,
// grad_indices); grad_indices carries no gradient).
//
// For query row (b,s) and selected slot j with key t = idx[j] inside the row's
// visible range and g = grad[j], with x_h = q[s,b,h,:] . k[t,b,:]:
//     dw[s,b,h]   += g * act(x_h)
//     P_h          = g * w[s,b,h] * act'(x_h)          (ReLU'(0) = 0)
//     dq[s,b,h,:] += P_h * k[t,b,:]
//     dk[t,b,:]   += sum_h P_h * q[s,b,h,:]
//
// Four launches, all on the caller's stream:
//   1. bwd_scatter_kernel: the selected grads become a dense G[b,s,t] (0 where
//      nothing is selected; slots outside the row's range are dropped).
//   2. bwd_tile_kernel<H, 0, D128>, query-major.  A persistent CTA takes tiles of
//      128 (query, head) rows and sweeps their visible keys 128 at a time:
//        X = Q K^T                 tcgen05, bf16 -> fp32 into TMEM
//        P = G w act'(X), dw += G act(X)   epilogue warps, one TMEM lane each;
//            P goes back into the same TMEM columns as bf16 hi + lo halves
//        dq += P_hi K + P_lo K     tcgen05 with A read from TMEM, K as an
//                                  MN-major operand of the same shared tile
//      dq and dw are written once per row tile.
//   3. bwd_tile_kernel<H, 1, D128>, key-major: the same pipeline with the roles of
//      the operands swapped -- a tile of 128 keys sweeps a chunk of query tiles
//      (128 (query, head) columns each), X^T = K Q^T, P^T, dk += P^T Q -- and
//      writes one partial dk per (key tile, chunk).
//   4. bwd_reduce_kernel: dk = each key tile's partials summed in a fixed order.
// No atomic operation touches dq, dk or dw: the results are deterministic.
//
// P is split into two bf16 halves (hi = bf16(P), lo = bf16(P - hi)) because the
// tensor cores multiply bf16 by bf16; together they carry about 16 bits of P.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lidx {

constexpr int kBT = 128;                           // rows of a tile; columns of X
constexpr int kBStages = 3;                        // streamed-tile ring
constexpr int kBRegions = 3;                       // X/P regions in TMEM, 128 columns each
// The second product of a tile is issued after the X product of the next tile,
// so the epilogue of one tile overlaps the X product of the next.  (Issuing two
// X products ahead measured slower.)  Two resident tiles then suffice.
constexpr int kBLookahead = 1;
constexpr int kBRes = 2;
constexpr int kBEpiWarps = 8;                      // two per TMEM lane quadrant, 64 columns each
constexpr int kBThreads = 64 + 32 * kBEpiWarps;
constexpr int kBMaxKeyTiles = 512;                 // Skv <= 65536
constexpr int kBMaxChunks = 512;                   // chunks of query tiles (key-major)
constexpr uint32_t kBTileBytes = kBT * 128;        // one 64-wide block of a 128-row tile

struct BwdParams {
    int B, S, Skv, H, D, Dp, ratio, act, grad_dtype;
    const int32_t* ks;  // nullable with ke: causal ranges from ratio
    const int32_t* ke;
    const float* w;     // [S,B,H]
    const float* G;     // [B,S,Skv_pad] dense selected grads
    int Skv_pad;
    void* dq;           // [S,B,H,D] fp32 or bf16
    float* dw;          // [S,B,H]
    float* part;        // [B*U][128][Dp] partial dk
    int qtiles, ntk, QT, nkb;
    int num_units;
    int U, CH, nchunks; // key-major: units per batch, query tiles per chunk, chunks
    uint64_t wait_ns;
    int debug_stall;    // 1: the TMA producer issues nothing (failure-detection tests)
    int cpre[kBMaxChunks + 1];   // key-major: first unit of each chunk within a batch
};

__device__ __forceinline__ void bwd_row_range(const BwdParams& p, int s, int& lo, int& hi) {
    if (p.ks == nullptr) {
        lo = 0;
        const long long e = (long long)(s + 1) / p.ratio;
        hi = (int)(e < p.Skv ? e : p.Skv);
    } else {
        lo = p.ks[s] > 0 ? p.ks[s] : 0;
        hi = p.ke[s] < p.Skv ? p.ke[s] : p.Skv;
        if (hi < lo) hi = lo;
    }
}

// Union [lo, hi) of the visible ranges of query tile qt's rows (empty: hi <= lo).
__device__ __forceinline__ void qtile_range(const BwdParams& p, int qt, int& lo, int& hi) {
    const int s0 = qt * p.QT, s1 = min(s0 + p.QT, p.S) - 1;
    if (p.ks == nullptr) {
        bwd_row_range(p, s1, lo, hi);
        return;
    }
    lo = p.Skv;
    hi = 0;
    for (int s = s0; s <= s1; ++s) {
        int a, e;
        bwd_row_range(p, s, a, e);
        if (e > a) {
            lo = min(lo, a);
            hi = max(hi, e);
        }
    }
}

// First query tile whose rows can see key tile kt (0 for explicit ranges).
__host__ __device__ __forceinline__ int bwd_qlo(bool causal, int kt, int ratio, int QT) {
    if (!causal) return 0;
    const long long s_min = ((long long)kt * kBT + 1) * ratio - 1;  // first row seeing key kt*128
    return (int)(s_min / QT);
}

struct BUnit {
    int b, res;         // batch; resident tile (query tile for MODE 0, key tile for MODE 1)
    int first, last;    // streamed tiles [first, last) (key tiles, or query tiles)
};

template <int MODE>
__device__ __forceinline__ BUnit bwd_unit(const BwdParams& p, int u) {
    BUnit un;
    if constexpr (MODE == 0) {
        un.res = p.qtiles - 1 - u / p.B;  // heaviest (latest) query tiles first
        un.b = u % p.B;
        int lo, hi;
        qtile_range(p, un.res, lo, hi);
        if (hi > lo) {
            un.first = lo / kBT;
            un.last = (hi + kBT - 1) / kBT;
        } else {
            un.first = un.last = 0;
        }
    } else {
        // chunk-major: the units of one chunk (one per key tile) cover the same
        // query tiles, so CTAs that run them at the same time share those tiles in L2
        un.b = u / p.U;
        const int r = u % p.U;
        int a = 0, z = p.nchunks - 1;  // last chunk whose first unit is <= r
        while (a < z) {
            const int mid = (a + z + 1) >> 1;
            if (p.cpre[mid] <= r)
                a = mid;
            else
                z = mid - 1;
        }
        un.res = r - p.cpre[a];
        un.first = max(a * p.CH, bwd_qlo(p.ks == nullptr, un.res, p.ratio, p.QT));
        un.last = min((a + 1) * p.CH, p.qtiles);
    }
    return un;
}

// Streamed tile x of unit un has work.
template <int MODE>
__device__ __forceinline__ bool bwd_active(const BwdParams& p, const BUnit& un, int x) {
    if constexpr (MODE == 0) return true;
    int lo, hi;
    qtile_range(p, x, lo, hi);
    return hi > lo && hi > un.res * kBT && lo < un.res * kBT + kBT;
}

template <int MODE>
__device__ __forceinline__ int bwd_count(const BwdParams& p, const BUnit& un) {
    if constexpr (MODE == 0) return un.last - un.first;
    int n = 0;
    for (int x = un.first; x < un.last; ++x) n += bwd_active<MODE>(p, un, x);
    return n;
}

// i-th unit of this CTA in snake order, -1 to skip, -2 past the end
__device__ __forceinline__ int bwd_unit_of(int i, int num_units) {
    const int G = gridDim.x;
    const int base = i * G;
    if (base >= num_units) return -2;
    const int u = base + ((i & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
    return u < num_units ? u : -1;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo_elem, float hi_elem) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
    return r;
}

// Packed fp32 pairs: each lane of the pair rounded as the scalar operation rounds.
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mov.b64 d, {%0, %1};\n\tfma.rn.f32x2 d, a, b, d;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// P of 32 columns -> packed bf16 hi and lo halves (element 2c in the low half).
// P - hi is exact in fp32, so lo carries the next 8 bits of P.
__device__ __forceinline__ void split_hi_lo(const float (&P)[32], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const uint32_t h2 = bf16x2_rn(P[2 * c], P[2 * c + 1]);
        hi[c] = h2;
        float r0, r1;
        sub2(r0, r1, P[2 * c], P[2 * c + 1], __uint_as_float(h2 << 16), __uint_as_float(h2 & 0xffff0000u));
        lo[c] = bf16x2_rn(r0, r1);
    }
}

// D128: D = 128 and ReLU, so that the shared-memory layout, the column loops and
// the activation are constant (other calls take D128 = false)
template <int H, int MODE, bool D128>
__global__ void __launch_bounds__(kBThreads, 1)
    bwd_tile_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmw,
                    const __grid_constant__ BwdParams p) {
    constexpr int QT = kBT / H;  // queries per tile of 128 (query, head) rows
    // With at least 8 heads, each stage also carries the tile's grads G [QT][128]
    // (and, key-major, its weights [QT][H]), loaded by TMA with the operand.
    constexpr bool kStaged = H >= 8;
    constexpr uint32_t kGBytes = kStaged ? QT * kBT * 4 : 0;
    constexpr uint32_t kWBytes = (kStaged && MODE == 1) ? QT * H * 4 : 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nkb = D128 ? 2 : p.nkb;
    const int Dp = D128 ? 128 : p.Dp, D = D128 ? 128 : p.D;
    const uint32_t tile_bytes = kBTileBytes * nkb;
    const uint32_t stage_bytes = tile_bytes + (kGBytes + kWBytes + 1023u) / 1024u * 1024u;
    uint8_t* sRes = smem;                          // [kBRes] resident tiles
    uint8_t* sStg = smem + kBRes * tile_bytes;     // [kBStages] streamed tiles (+ G, w)
    float* sDw = (float*)(sStg + kBStages * stage_bytes);  // [2][128] dw partials of column half 1
    uint64_t* bars = (uint64_t*)(sDw + 2 * 4 * kBT);
    uint64_t* res_full = bars;                     // [kBRes]
    uint64_t* res_empty = bars + kBRes;            // [kBRes]
    uint64_t* k_full = bars + 2 * kBRes;           // [kBStages]
    uint64_t* k_empty = k_full + kBStages;         // [kBStages]
    uint64_t* x_full = k_empty + kBStages;         // [kBRegions]
    uint64_t* p_full = x_full + kBRegions;         // [kBRegions]
    uint64_t* r_free = p_full + kBRegions;         // [kBRegions]
    uint64_t* acc_full = r_free + kBRegions;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* dw_full = acc_empty + 1;             // [2] column quarters 1..3 -> quarter 0
    uint64_t* dw_empty = dw_full + 2;              // [2] quarter 0 -> quarters 1..3
    uint32_t* tmem_slot = (uint32_t*)(dw_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kBRes; ++i) {
            mbar_init(res_full + i, 1);
            mbar_init(res_empty + i, 1);
        }
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(k_full + i, 1);
            mbar_init(k_empty + i, 1);
        }
        for (int i = 0; i < kBRegions; ++i) {
            mbar_init(x_full + i, 1);
            mbar_init(p_full + i, kBEpiWarps);
            mbar_init(r_free + i, 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kBEpiWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(dw_full + i, kBEpiWarps / 2);
            mbar_init(dw_empty + i, kBEpiWarps / 2);
        }
        fence_mbar_init();
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        if constexpr (kStaged) tma_prefetch_desc(&tmg);
        if constexpr (kStaged && MODE == 1) tma_prefetch_desc(&tmw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t acc_col = kBRegions * kBT;  // columns [384, 384 + Dp)

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && !p.debug_stall) {
            int kcount = 0, ucount = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int u = bwd_unit_of(i, p.num_units);
                if (u == -2) break;
                if (u < 0) continue;
                const BUnit un = bwd_unit<MODE>(p, u);
                if (bwd_count<MODE>(p, un) == 0) continue;
                const int ub = ucount % kBRes;
                if (!(ok = mbar_wait(res_empty + ub, ((ucount / kBRes) & 1) ^ 1, p.wait_ns))) break;
                ++ucount;
                mbar_arrive_expect_tx(res_full + ub, tile_bytes);
                for (int kb = 0; kb < nkb; ++kb) {
                    uint8_t* dst = sRes + ub * tile_bytes + kb * kBTileBytes;
                    if constexpr (MODE == 0)  // q [S,B,H,D]: dims (D, H, B, S)
                        tma_load_4d(dst, &tmq, res_full + ub, kb * 64, 0, un.b, un.res * QT);
                    else  // k [Skv,B,D]: dims (D, B, Skv)
                        tma_load_3d(dst, &tmk, res_full + ub, kb * 64, un.b, un.res * kBT);
                }
                for (int x = un.first; x < un.last && ok; ++x) {
                    if (!bwd_active<MODE>(p, un, x)) continue;
                    const int st = kcount % kBStages;
                    if (!(ok = mbar_wait(k_empty + st, ((kcount / kBStages) & 1) ^ 1, p.wait_ns))) break;
                    ++kcount;
                    mbar_arrive_expect_tx(k_full + st, tile_bytes + kGBytes + kWBytes);
                    uint8_t* sdst = sStg + st * stage_bytes;
                    for (int kb = 0; kb < nkb; ++kb) {
                        uint8_t* dst = sdst + kb * kBTileBytes;
                        if constexpr (MODE == 0)
                            tma_load_3d(dst, &tmk, k_full + st, kb * 64, un.b, x * kBT);
                        else
                            tma_load_4d(dst, &tmq, k_full + st, kb * 64, 0, un.b, x * QT);
                    }
                    if constexpr (kStaged) {  // G [B,S,Skv_pad]: dims (Skv_pad, S, B)
                        if constexpr (MODE == 0)
                            tma_load_3d(sdst + tile_bytes, &tmg, k_full + st, x * kBT, un.res * QT, un.b);
                        else
                            tma_load_3d(sdst + tile_bytes, &tmg, k_full + st, un.res * kBT, x * QT, un.b);
                    }
                    if constexpr (kStaged && MODE == 1)  // w [S,B,H]: dims (H, B, S)
                        tma_load_3d(sdst + tile_bytes + kGBytes, &tmw, k_full + st, 0, un.b, x * QT);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_x = idesc_bf16_f32(kBT, kBT);
            const uint32_t idesc_2 = idesc_bf16_f32(kBT, (uint32_t)Dp) | (1u << 16);  // B MN-major
            const int nk = Dp / 16;
            // base descriptors of every buffer; a k-step adds its byte offset / 16 to the
            // 14-bit start-address field (shared addresses stay below 256 KB: no carry)
            uint64_t rd[kBRes], sd[kBStages], md[kBStages];
#pragma unroll
            for (int j = 0; j < kBRes; ++j) rd[j] = smem_desc_kmajor(smem_u32(sRes + j * tile_bytes), 128);
#pragma unroll
            for (int j = 0; j < kBStages; ++j) {
                sd[j] = smem_desc_kmajor(smem_u32(sStg + j * stage_bytes), 128);
                md[j] = smem_desc_mn_sw128(smem_u32(sStg + j * stage_bytes), kBTileBytes);
            }
            auto koff16 = [](int k) {  // K-major k-step: 64-wide block, then 32 bytes per 16
                return (uint64_t)((((k * 16) / 64) * kBTileBytes + ((k * 16) % 64) * 2) >> 4);
            };
            struct Pend {
                int r, st, ub, tc, uc;
                bool first, last;
            };
            bool ok = true;
            // by value: a reference kept the queue in local memory
            auto second = [&](const Pend t) -> bool {
                if (!mbar_wait(p_full + t.r, (t.tc / kBRegions) & 1, p.wait_ns)) return false;
                if (t.first && !mbar_wait(acc_empty, (t.uc & 1) ^ 1, p.wait_ns)) return false;
                tc_fence_after();
                const uint32_t a0 = tmem_base + t.r * kBT;
                uint64_t b0 = md[0];
#pragma unroll
                for (int j = 1; j < kBStages; ++j) b0 = t.st == j ? md[j] : b0;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t b = b0 + (uint64_t)((kk * 16 * 128) >> 4);  // 16 rows per step
                    const uint32_t a = a0 + 32 * (kk >> 1) + 8 * (kk & 1);
                    umma_f16_ts(tmem_base + acc_col, a, b, idesc_2, (t.first && kk == 0) ? 0u : 1u);
                    umma_f16_ts(tmem_base + acc_col, a + 16, b, idesc_2, 1u);
                }
                umma_commit(r_free + t.r);
                umma_commit(k_empty + t.st);
                if (t.last) {
                    umma_commit(acc_full);
                    umma_commit(res_empty + t.ub);
                }
                return true;
            };
            Pend queue[kBLookahead];
            int nq = 0;
            int kcount = 0, tcount = 0, ucount = 0;
            for (int i = 0; ok; ++i) {
                const int u = bwd_unit_of(i, p.num_units);
                if (u == -2) break;
                if (u < 0) continue;
                const BUnit un = bwd_unit<MODE>(p, u);
                const int n = bwd_count<MODE>(p, un);
                if (n == 0) continue;
                const int ub = ucount % kBRes, uc = ucount;
                if (!(ok = mbar_wait(res_full + ub, (ucount / kBRes) & 1, p.wait_ns))) break;
                ++ucount;
                int idx = 0;
                for (int x = un.first; x < un.last; ++x) {
                    if (!bwd_active<MODE>(p, un, x)) continue;
                    const int st = kcount % kBStages, r = tcount % kBRegions;
                    if (!(ok = mbar_wait(k_full + st, (kcount / kBStages) & 1, p.wait_ns))) break;
                    if (!(ok = mbar_wait(r_free + r, ((tcount / kBRegions) & 1) ^ 1, p.wait_ns))) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + r * kBT;
                    uint64_t a0 = rd[0];
#pragma unroll
                    for (int j = 1; j < kBRes; ++j) a0 = ub == j ? rd[j] : a0;
                    uint64_t b0 = sd[0];
#pragma unroll
                    for (int j = 1; j < kBStages; ++j) b0 = st == j ? sd[j] : b0;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (k < nk) umma_f16(d, a0 + koff16(k), b0 + koff16(k), idesc_x, k > 0 ? 1u : 0u);
                    umma_commit(x_full + r);
                    if (nq == kBLookahead) {
                        if (!(ok = second(queue[0]))) break;
#pragma unroll
                        for (int j = 1; j < kBLookahead; ++j) queue[j - 1] = queue[j];
                        --nq;
                    }
                    // constant indices keep the queue in registers
                    const Pend pend{r, st, ub, tcount, uc, idx == 0, idx == n - 1};
#pragma unroll
                    for (int j = 0; j < kBLookahead; ++j)
                        if (j == nq) queue[j] = pend;
                    ++nq;
                    ++kcount;
                    ++tcount;
                    ++idx;
                }
            }
#pragma unroll
            for (int j = 0; j < kBLookahead; ++j)
                if (ok && j < nq) ok = second(queue[j]);
        }
    } else {
        // --------------------------------------------------------- epilogue
        // Two warps share each TMEM lane quadrant: warp half chalf takes columns
        // [64*chalf, 64*chalf + 64) of X and of the accumulator.
        const int quad = warp & 3;           // TMEM lane quadrant this warp may read
        const int chalf = (warp - 2) >> 2;
        const int row = quad * 32 + lane;    // TMEM lane = row of the resident tile
        const uint32_t lane_addr = tmem_base + ((uint32_t)(quad * 32) << 16);
        int tcount = 0, ucount = 0, done_units = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            const int u = bwd_unit_of(i, p.num_units);
            if (u == -2) break;
            if (u < 0) continue;
            const BUnit un = bwd_unit<MODE>(p, u);
            const int n = bwd_count<MODE>(p, un);
            // this thread's output row
            int s = 0, h = 0, t = 0;
            bool rvalid;
            if constexpr (MODE == 0) {
                s = un.res * QT + row / H;
                h = row % H;
                rvalid = s < p.S;
            } else {
                t = un.res * kBT + row;
                rvalid = true;  // partial rows past Skv are written and never read
            }
            const float wv = (MODE == 0 && rvalid) ? p.w[((size_t)s * p.B + un.b) * H + h] : 0.f;
            float dw4[4] = {0.f, 0.f, 0.f, 0.f};
            if (n > 0) {
                for (int x = un.first; x < un.last; ++x) {
                    if (!bwd_active<MODE>(p, un, x)) continue;
                    const int r = tcount % kBRegions;
                    const float* gS = (const float*)(sStg + (tcount % kBStages) * stage_bytes + tile_bytes);
                    const float* wS = gS + QT * kBT;
                    const int tc = tcount++;
                    if (!(ok = mbar_wait(x_full + r, (tc / kBRegions) & 1, p.wait_ns))) break;
                    tc_fence_after();
#pragma unroll
                    for (int cc = 2 * chalf; cc < 2 * chalf + 2; ++cc) {
                    const int c = cc;
                    uint32_t xr[32];
                    tmem_ld32(lane_addr + r * kBT + 32 * c, xr);
                    float P[32];
                    if constexpr (MODE == 0) {
                        // columns = keys x*128 + 32c + i of this thread's query row
                        float g[32];
                        if (rvalid) {
                            const float4* g4 = reinterpret_cast<const float4*>(
                                kStaged ? gS + (row / H) * kBT + 32 * c
                                        : p.G + ((size_t)un.b * p.S + s) * p.Skv_pad + (size_t)x * kBT +
                                              32 * c);
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const float4 q4 = g4[v];
                                g[4 * v] = q4.x;
                                g[4 * v + 1] = q4.y;
                                g[4 * v + 2] = q4.z;
                                g[4 * v + 3] = q4.w;
                            }
                        } else {
#pragma unroll
                            for (int v = 0; v < 32; ++v) g[v] = 0.f;
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int v = 0; v < 32; v += 2) {
                            const float x0 = __uint_as_float(xr[v]), x1 = __uint_as_float(xr[v + 1]);
                            const bool relu = D128 || p.act == 0;
                            const float a0 = relu ? fmaxf(x0, 0.f) : x0, a1 = relu ? fmaxf(x1, 0.f) : x1;
                            fma2(dw4[v & 3], dw4[(v & 3) + 1], g[v], g[v + 1], a0, a1);
                            float p0, p1;
                            mul2(p0, p1, g[v], g[v + 1], wv, wv);
                            P[v] = (!relu || x0 > 0.f) ? p0 : 0.f;
                            P[v + 1] = (!relu || x1 > 0.f) ? p1 : 0.f;
                        }
                    } else {
                        // columns = (query, head) 32c + i of query tile x; this thread's key t
                        float gw[32];
                        if constexpr (kStaged) {
                            // the stage holds this query tile's grads [QT][128] and weights
                            // [QT][H] (zero past S): columns 32c .. 32c + 31
#pragma unroll
                            for (int v = 0; v < 32; v += 4) {
                                const float4 w4 = *reinterpret_cast<const float4*>(wS + 32 * c + v);
                                const float wv4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                for (int e = 0; e < 4; e += 2)
                                    mul2(gw[v + e], gw[v + e + 1], gS[((32 * c + v + e) / H) * kBT + row],
                                         gS[((32 * c + v + e + 1) / H) * kBT + row], wv4[e], wv4[e + 1]);
                            }
                        } else {
#pragma unroll
                            for (int v = 0; v < 32; ++v) {
                                const int col = 32 * c + v;
                                const int sq = x * QT + col / H, hq = col % H;
                                gw[v] = sq < p.S ? p.G[((size_t)un.b * p.S + sq) * p.Skv_pad + t] *
                                                       p.w[((size_t)sq * p.B + un.b) * H + hq]
                                                 : 0.f;
                            }
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int v = 0; v < 32; ++v) {
                            const float xv = __uint_as_float(xr[v]);
                            P[v] = (D128 || p.act == 0) ? (xv > 0.f ? gw[v] : 0.f) : gw[v];
                        }
                    }
                    uint32_t hi[16], lo[16];
                    split_hi_lo(P, hi, lo);
                    tmem_st16(lane_addr + r * kBT + 32 * c, hi);
                    tmem_st16(lane_addr + r * kBT + 32 * c + 16, lo);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full + r);
                }
                if (!ok) break;
            }
            // outputs of the unit: this warp's 64 columns of the accumulator, 32 at a time
            if (n > 0) {
                if (!(ok = mbar_wait(acc_full, ucount & 1, p.wait_ns))) break;
                ++ucount;
                tc_fence_after();
            }
#pragma unroll 1
            for (int c = 2 * chalf; c < 2 * chalf + 2; ++c) {
            float out[32];
            if (n > 0 && 32 * c < Dp) {
                uint32_t ar[32];
                tmem_ld32(lane_addr + acc_col + 32 * c, ar);
                tmem_ld_wait();
#pragma unroll
                for (int v = 0; v < 32; ++v) out[v] = __uint_as_float(ar[v]);
            } else {
#pragma unroll
                for (int v = 0; v < 32; ++v) out[v] = 0.f;
            }
            const int d0 = 32 * c;
            const int dn = min(32, D - d0);  // valid output columns of this chunk
            if constexpr (MODE == 0) {
                if (rvalid && dn > 0) {
                    const size_t o = (((size_t)s * p.B + un.b) * H + h) * D + d0;
                    if (p.grad_dtype == 0) {
                        float* dst = (float*)p.dq + o;
                        if (dn == 32) {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                reinterpret_cast<float4*>(dst)[v] =
                                    make_float4(out[4 * v], out[4 * v + 1], out[4 * v + 2], out[4 * v + 3]);
                        } else {  // ragged last chunk; constant indices keep `out` in registers
#pragma unroll
                            for (int v = 0; v < 32; ++v)
                                if (v < dn) dst[v] = out[v];
                        }
                    } else {
                        uint16_t* dst = (uint16_t*)p.dq + o;
                        if (dn == 32) {
                            uint32_t pk[16];
#pragma unroll
                            for (int v = 0; v < 16; ++v) pk[v] = bf16x2_rn(out[2 * v], out[2 * v + 1]);
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                reinterpret_cast<uint4*>(dst)[v] =
                                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                        } else {
#pragma unroll
                            for (int v = 0; v < 32; ++v)
                                if (v < dn) dst[v] = (uint16_t)(bf16x2_rn(out[v], 0.f) & 0xffffu);
                        }
                    }
                }
            } else {
                if (dn > 0 && d0 < Dp) {
                    float* dst = p.part + ((size_t)u * kBT + row) * Dp + d0;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        reinterpret_cast<float4*>(dst)[v] =
                            make_float4(out[4 * v], out[4 * v + 1], out[4 * v + 2], out[4 * v + 3]);
                }
            }
            }
            if (n > 0) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            if constexpr (MODE == 0) {
                // dw: the two column halves' partial sums, added in a fixed order;
                // half 1 hands its partial to half 0 through a double buffer
                const float dw_acc = (dw4[0] + dw4[1]) + (dw4[2] + dw4[3]);
                const int db = done_units & 1;
                const uint32_t dph = (done_units >> 1) & 1;
                float* dwb = sDw + db * kBT;
                if (chalf == 1) {
                    if (!(ok = mbar_wait(dw_empty + db, dph ^ 1, p.wait_ns))) break;
                    dwb[row] = dw_acc;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dw_full + db);
                } else {
                    if (!(ok = mbar_wait(dw_full + db, dph, p.wait_ns))) break;
                    const float o1 = dwb[row];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dw_empty + db);
                    if (rvalid) p.dw[((size_t)s * p.B + un.b) * H + h] = dw_acc + o1;
                }
            }
            ++done_units;
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

// Dense selected grads: G[b,s,t] = sum of grad[b,s,j] over slots j with
// idx[b,s,j] = t inside the row's visible range; 0 elsewhere.  One CTA per row
// at a time; the row is built in shared memory when it fits.
constexpr int kScatterThreads = 256;
constexpr int kScatterK = 4;  // slots a thread holds ahead: rows of up to 1024 selected keys

__global__ void __launch_bounds__(kScatterThreads)
    bwd_scatter_kernel(const int32_t* __restrict__ idx, const float* __restrict__ grad, int B, int S,
                       int Skv, int Skv_pad, int ratio, const int32_t* __restrict__ ksa,
                       const int32_t* __restrict__ kea, int topk, float* __restrict__ G, int in_smem) {
    extern __shared__ __align__(16) float srow[];
    const int tid = threadIdx.x;
    const int rows = B * S;
    // The next row's slots are loaded while this row is built, so that their latency
    // overlaps the zeroing, the atomics and the write-out (rows of up to
    // kScatterK * kScatterThreads slots; longer rows load their slots in place).
    // Measured on the backward workload (1024 slots a row): 0.986 -> 0.972 ms.
    const bool ahead = topk <= kScatterK * kScatterThreads;
    int nt[kScatterK];
    float ng[kScatterK];
#pragma unroll
    for (int k = 0; k < kScatterK; ++k) {
        const int j = tid + k * kScatterThreads, r = blockIdx.x;
        const bool ok = ahead && r < rows && j < topk;
        nt[k] = ok ? idx[(size_t)r * topk + j] : -1;
        ng[k] = ok ? grad[(size_t)r * topk + j] : 0.f;
    }
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        int ct[kScatterK];
        float cg[kScatterK];
#pragma unroll
        for (int k = 0; k < kScatterK; ++k) {
            ct[k] = nt[k];
            cg[k] = ng[k];
            const int j = tid + k * kScatterThreads, rn = r + gridDim.x;
            const bool ok = ahead && rn < rows && j < topk;
            nt[k] = ok ? idx[(size_t)rn * topk + j] : -1;
            ng[k] = ok ? grad[(size_t)rn * topk + j] : 0.f;
        }
        const int s = r % S;
        int lo, hi;
        if (ksa == nullptr) {
            lo = 0;
            const long long e = (long long)(s + 1) / ratio;
            hi = (int)(e < Skv ? e : Skv);
        } else {
            lo = ksa[s] > 0 ? ksa[s] : 0;
            hi = kea[s] < Skv ? kea[s] : Skv;
        }
        float* grow = G + (size_t)r * Skv_pad;
        float* dst = in_smem ? srow : grow;
        __syncthreads();  // the previous row is written out
        for (int t = tid * 4; t < Skv_pad; t += kScatterThreads * 4)
            *reinterpret_cast<float4*>(dst + t) = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
        if (ahead) {
#pragma unroll
            for (int k = 0; k < kScatterK; ++k)
                if (ct[k] >= lo && ct[k] < hi) atomicAdd(dst + ct[k], cg[k]);
        } else {
            const int32_t* irow = idx + (size_t)r * topk;
            const float* gr = grad + (size_t)r * topk;
            for (int j = tid; j < topk; j += kScatterThreads) {
                const int t = irow[j];
                if (t >= lo && t < hi) atomicAdd(dst + t, gr[j]);
            }
        }
        if (in_smem) {
            __syncthreads();
            for (int t = tid * 4; t < Skv_pad; t += kScatterThreads * 4)
                *reinterpret_cast<float4*>(grow + t) = *reinterpret_cast<const float4*>(srow + t);
        }
    }
}

// First partial-dk unit of each chunk of query tiles within a batch.
struct ChunkTable {
    int cpre[kBMaxChunks + 1];
};

// Chunk of the first query tile that sees key tile kt, or nchunks when none does.
__host__ __device__ __forceinline__ int bwd_c0(bool causal, int kt, int ratio, int QT, int qtiles,
                                               int CH, int nchunks) {
    const int qlo = bwd_qlo(causal, kt, ratio, QT);
    return qlo < qtiles ? qlo / CH : nchunks;
}

// dk[t,b,:] = sum over the chunks c of key tile t/128 of part[unit(b, c, t/128)][t%128][:],
// in a fixed order: the chunk range is cut into kReduceSplit runs, each summed in chunk
// order by its own thread, and the run sums are added pairwise ((r0 + r1) + (r2 + r3)).
// A block takes kReduceOut outputs (4 columns each) at a time, so that enough loads are
// in flight for a sum over only tens of chunks.
constexpr int kReduceSplit = 4, kReduceOut = 64, kReduceThreads = kReduceSplit * kReduceOut;

__global__ void __launch_bounds__(kReduceThreads)
    bwd_reduce_kernel(const float* __restrict__ part, int B, int Skv, int D, int Dp, int U,
                      const __grid_constant__ ChunkTable tab, int nchunks, int CH, int QT, int qtiles,
                      int ratio, int causal, int grad_dtype, void* dk) {
    __shared__ float4 runs[kReduceSplit][kReduceOut];
    const int D4 = D / 4;
    const int64_t n = (int64_t)B * Skv * D4;
    const int64_t ngroups = (n + kReduceOut - 1) / kReduceOut;
    const int o_local = threadIdx.x % kReduceOut, q = threadIdx.x / kReduceOut;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const int64_t e = g * kReduceOut + o_local;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int t = 0, b = 0, d4 = 0;
        if (e < n) {
            d4 = (int)(e % D4) * 4;
            const int64_t bt = e / D4;
            t = (int)(bt % Skv);
            b = (int)(bt / Skv);
            const int kt = t / kBT, tl = t % kBT;
            const int c0 = bwd_c0(causal != 0, kt, ratio, QT, qtiles, CH, nchunks), len = nchunks - c0;
            const int ca = c0 + (int)((int64_t)len * q / kReduceSplit);
            const int cb = c0 + (int)((int64_t)len * (q + 1) / kReduceSplit);
            // one accumulator in chunk order; the unrolling only keeps loads in flight
#pragma unroll 4
            for (int c = ca; c < cb; ++c) {
                const int u = b * U + tab.cpre[c] + kt;
                const float4 v = *reinterpret_cast<const float4*>(part + ((size_t)u * kBT + tl) * Dp + d4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
        }
        runs[q][o_local] = acc;
        __syncthreads();
        if (q == 0 && e < n) {
            const float4 r1 = runs[1][o_local], r2 = runs[2][o_local], r3 = runs[3][o_local];
            static_assert(kReduceSplit == 4, "pairwise combination of four runs");
            float4 sum;
            sum.x = (acc.x + r1.x) + (r2.x + r3.x);
            sum.y = (acc.y + r1.y) + (r2.y + r3.y);
            sum.z = (acc.z + r1.z) + (r2.z + r3.z);
            sum.w = (acc.w + r1.w) + (r2.w + r3.w);
            const size_t o = ((size_t)t * B + b) * D + d4;
            if (grad_dtype == 0) {
                *reinterpret_cast<float4*>((float*)dk + o) = sum;
            } else {
                const uint32_t lo = bf16x2_rn(sum.x, sum.y), hi = bf16x2_rn(sum.z, sum.w);
                *reinterpret_cast<uint2*>((uint16_t*)dk + o) = make_uint2(lo, hi);
            }
        }
        __syncthreads();  // runs[] is reused by the next group
    }
}

// ------------------------------------------------------------------- host
LIDX_STATUS_READER(status_bwd)

struct BwdPlan {
    int Dp, QT, qtiles, ntk, Skv_pad, CH, U, nkb, nchunks;
    size_t g_bytes, part_bytes;
    int cpre[kBMaxChunks + 1];
};

// Tiling of the backward.  Key-major units: chunk c of query tiles [c*CH, (c+1)*CH)
// holds one unit per key tile that some row of the chunk sees; `causal` gives each
// key tile its first visible query tile (explicit ranges: every tile).
static void bwd_plan(int64_t B, int64_t S, int64_t Skv, int H, int D, int ratio, bool causal, int sms,
                     BwdPlan& pl) {
    pl.Dp = (D + 63) / 64 * 64;
    pl.nkb = pl.Dp / 64;
    pl.QT = kBT / H;
    pl.qtiles = (int)((S + pl.QT - 1) / pl.QT);
    pl.ntk = (int)((Skv + kBT - 1) / kBT);
    pl.Skv_pad = pl.ntk * kBT;
    int64_t T = 0;  // (query tile, key tile) pairs
    for (int kt = 0; kt < pl.ntk; ++kt) {
        const int qlo = bwd_qlo(causal, kt, ratio, pl.QT);
        T += qlo < pl.qtiles ? pl.qtiles - qlo : 0;
    }
    T *= B;
    const int64_t target = 4 * (int64_t)sms;  // about four units per SM
    pl.CH = (int)((T + target - 1) / target);
    const int ch_min = (pl.qtiles + kBMaxChunks - 1) / kBMaxChunks;
    if (pl.CH < ch_min) pl.CH = ch_min;
    if (pl.CH < 1) pl.CH = 1;
    pl.nchunks = (pl.qtiles + pl.CH - 1) / pl.CH;
    int U = 0, kt = 0;
    for (int c = 0; c < pl.nchunks; ++c) {
        while (kt < pl.ntk && bwd_c0(causal, kt, ratio, pl.QT, pl.qtiles, pl.CH, pl.nchunks) <= c) ++kt;
        pl.cpre[c] = U;
        U += kt;  // key tiles 0 .. kt-1 have a unit in chunk c
    }
    pl.cpre[pl.nchunks] = U;
    pl.U = U;
    pl.g_bytes = ((size_t)B * S * pl.Skv_pad * 4 + 255) / 256 * 256;
    pl.part_bytes = (size_t)B * U * kBT * pl.Dp * 4;
}

// Units per batch are sum over key tiles of (chunks from its first one on) <=
// T/(B*CH) + 2*ntk, and T/CH <= 4*sms: the bound holds for causal and
// explicit-range calls alike.
size_t bwd_workspace_bytes(int64_t B, int64_t S, int64_t Skv, int H, int D, int topk, int num_sms) {
    (void)topk;
    if (B <= 0 || S <= 0 || Skv <= 0 || H < 1 || H > 128) return 0;
    const int64_t Dp = (D + 63) / 64 * 64;
    const int64_t ntk = (Skv + kBT - 1) / kBT;
    const size_t g = ((size_t)B * S * ntk * kBT * 4 + 255) / 256 * 256;
    const size_t units = (size_t)4 * num_sms + (size_t)2 * B * ntk;
    return g + units * kBT * Dp * 4;
}

static int encode_bwd_maps(const BwdLaunch& a, CUtensorMap* mq, CUtensorMap* mk, int QT) {
    const int H = a.H, D = a.D, B = a.B;
    cuuint32_t es[4] = {1, 1, 1, 1};
    // q [S,B,H,D]: dims (D, H, B, S); a 128-row tile = QT queries x H heads
    cuuint64_t qdim[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B, (cuuint64_t)a.S};
    cuuint64_t qstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)B * H * D * 2};
    cuuint32_t qbox[4] = {64, (cuuint32_t)H, 1, (cuuint32_t)QT};
    if (encode_tiled(mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)a.q, qdim, qstr, qbox, es,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return 1;
    // k [Skv,B,D]: dims (D, B, Skv)
    cuuint64_t kdim[3] = {(cuuint64_t)D, (cuuint64_t)B, (cuuint64_t)a.Skv};
    cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)B * D * 2};
    cuuint32_t kbox[3] = {64, 1, (cuuint32_t)kBT};
    if (encode_tiled(mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.k, kdim, kstr, kbox, es,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return 1;
    return 0;
}

// G [B,S,Skv_pad] fp32 as dims (Skv_pad, S, B), box [QT rows][128 keys]; w [S,B,H]
// fp32 as dims (H, B, S), box [QT queries][H].  Used when H >= 8.
static int encode_stage_maps(const BwdLaunch& a, const float* G, int Skv_pad, int QT, CUtensorMap* mg,
                             CUtensorMap* mw) {
    cuuint32_t es[3] = {1, 1, 1};
    cuuint64_t gdim[3] = {(cuuint64_t)Skv_pad, (cuuint64_t)a.S, (cuuint64_t)a.B};
    cuuint64_t gstr[2] = {(cuuint64_t)Skv_pad * 4, (cuuint64_t)a.S * Skv_pad * 4};
    cuuint32_t gbox[3] = {(cuuint32_t)kBT, (cuuint32_t)QT, 1};
    if (encode_tiled(mg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, (void*)G, gdim, gstr, gbox, es,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return 1;
    cuuint64_t wdim[3] = {(cuuint64_t)a.H, (cuuint64_t)a.B, (cuuint64_t)a.S};
    cuuint64_t wstr[2] = {(cuuint64_t)a.H * 4, (cuuint64_t)a.B * a.H * 4};
    cuuint32_t wbox[3] = {(cuuint32_t)a.H, 1, (cuuint32_t)QT};
    if (encode_tiled(mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, (void*)a.w, wdim, wstr, wbox, es,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return 1;
    return 0;
}

static size_t bwd_smem_bytes(int nkb, int H, int MODE) {
    const size_t tile = (size_t)kBTileBytes * nkb;
    size_t extra = 0;
    if (H >= 8) extra = ((size_t)(kBT / H) * kBT * 4 + (MODE == 1 ? (size_t)kBT * 4 : 0) + 1023) / 1024 * 1024;
    return 1024 + kBRes * tile + kBStages * (tile + extra) + 2 * 4 * kBT * 4 + 32 * 8 + 16;
}

template <int H, bool D128>
static cudaError_t bwd_tiles_hd(const CUtensorMap* maps, const BwdParams& p0, const BwdLaunch& a) {
    BwdParams p = p0;
    // dq and dw, query-major; at least 120 KB of shared memory so that one CTA
    // (and its 512 TMEM columns) owns each SM
    {
        int smem = (int)bwd_smem_bytes(p.nkb, H, 0);
        if (smem < 120 * 1024) smem = 120 * 1024;
        auto kern = bwd_tile_kernel<H, 0, D128>;
        cudaError_t e = set_smem_attr((const void*)kern, smem);
        if (e != cudaSuccess) return e;
        p.num_units = p.B * p.qtiles;
        const int grid = p.num_units < a.num_sms ? p.num_units : a.num_sms;
        if (grid > 0) kern<<<grid, kBThreads, smem, a.stream>>>(maps[0], maps[1], maps[2], maps[3], p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // partial dk, key-major
    {
        int smem = (int)bwd_smem_bytes(p.nkb, H, 1);
        if (smem < 120 * 1024) smem = 120 * 1024;
        auto kern = bwd_tile_kernel<H, 1, D128>;
        cudaError_t e = set_smem_attr((const void*)kern, smem);
        if (e != cudaSuccess) return e;
        p.num_units = p.B * p.U;
        const int grid = p.num_units < a.num_sms ? p.num_units : a.num_sms;
        if (grid > 0) kern<<<grid, kBThreads, smem, a.stream>>>(maps[0], maps[1], maps[2], maps[3], p);
        return cudaGetLastError();
    }
}

template <int H>
static cudaError_t bwd_tiles_h(const CUtensorMap* maps, const BwdParams& p, const BwdLaunch& a) {
    const bool d128 = p.D == 128 && p.act == 0;
    return d128 ? bwd_tiles_hd<H, true>(maps, p, a) : bwd_tiles_hd<H, false>(maps, p, a);
}

cudaError_t bwd_launch(const BwdLaunch& a) {
    const int64_t rows = (int64_t)a.B * a.S;
    const size_t es = a.grad_dtype ? 2 : 4;
    if (a.Skv == 0) {  // nothing visible: every gradient is zero
        cudaError_t e = cudaMemsetAsync(a.dq, 0, es * (size_t)rows * a.H * a.D, a.stream);
        if (e != cudaSuccess) return e;
        return cudaMemsetAsync(a.dw, 0, sizeof(float) * (size_t)rows * a.H, a.stream);
    }
    if ((a.Skv + kBT - 1) / kBT > kBMaxKeyTiles || a.H < 1 || a.H > 128) return cudaErrorInvalidValue;
    BwdPlan pl;
    bwd_plan(a.B, a.S, a.Skv, a.H, a.D, a.ratio, a.ks == nullptr, a.num_sms, pl);
    if (pl.g_bytes + pl.part_bytes > a.workspace_bytes) return cudaErrorInvalidValue;
    float* G = (float*)a.workspace;
    float* part = (float*)((uint8_t*)a.workspace + pl.g_bytes);

    // 1. dense selected grads
    {
        const size_t row_bytes = (size_t)pl.Skv_pad * 4;
        const int in_smem = row_bytes <= 64 * 1024;
        const int smem = in_smem ? (int)row_bytes : 0;
        if (in_smem) {
            cudaError_t e = set_smem_attr((const void*)bwd_scatter_kernel, smem);
            if (e != cudaSuccess) return e;
        }
        int64_t grid = (int64_t)a.num_sms * 8;  // eight rows in flight per SM
        if (grid > rows) grid = rows;
        bwd_scatter_kernel<<<(unsigned)grid, kScatterThreads, smem, a.stream>>>(
            a.idx, a.grad, a.B, a.S, a.Skv, pl.Skv_pad, a.ratio, a.ks, a.ke, a.topk, G, in_smem);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // 2, 3. tensor-core tiles
    CUtensorMap maps[4];
    if (encode_bwd_maps(a, &maps[0], &maps[1], pl.QT)) return cudaErrorInvalidValue;
    if (a.H >= 8) {
        if (encode_stage_maps(a, G, pl.Skv_pad, pl.QT, &maps[2], &maps[3])) return cudaErrorInvalidValue;
    } else {
        maps[2] = maps[0];  // not read
        maps[3] = maps[0];
    }
    BwdParams p;
    memset(&p, 0, sizeof p);
    p.B = a.B;
    p.S = a.S;
    p.Skv = a.Skv;
    p.H = a.H;
    p.D = a.D;
    p.Dp = pl.Dp;
    p.nkb = pl.nkb;
    p.ratio = a.ratio;
    p.act = a.act;
    p.grad_dtype = a.grad_dtype;
    p.ks = a.ks;
    p.ke = a.ke;
    p.w = a.w;
    p.G = G;
    p.Skv_pad = pl.Skv_pad;
    p.dq = a.dq;
    p.dw = a.dw;
    p.part = part;
    p.qtiles = pl.qtiles;
    p.ntk = pl.ntk;
    p.QT = pl.QT;
    p.U = pl.U;
    p.CH = pl.CH;
    p.nchunks = pl.nchunks;
    p.wait_ns = wait_limit_ns();
    p.debug_stall = debug_stall();
    memcpy(p.cpre, pl.cpre, sizeof(int) * (pl.nchunks + 1));
    cudaError_t e;
    switch (a.H) {
        case 1: e = bwd_tiles_h<1>(maps, p, a); break;
        case 2: e = bwd_tiles_h<2>(maps, p, a); break;
        case 4: e = bwd_tiles_h<4>(maps, p, a); break;
        case 8: e = bwd_tiles_h<8>(maps, p, a); break;
        case 16: e = bwd_tiles_h<16>(maps, p, a); break;
        case 32: e = bwd_tiles_h<32>(maps, p, a); break;
        case 64: e = bwd_tiles_h<64>(maps, p, a); break;
        case 128: e = bwd_tiles_h<128>(maps, p, a); break;
        default: e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    // 4. fixed-order reduction of the partial dk
    ChunkTable tab;
    memcpy(tab.cpre, pl.cpre, sizeof(int) * (pl.nchunks + 1));
    const int64_t n = (int64_t)a.B * a.Skv * (a.D / 4);
    int64_t grid = (n + kReduceOut - 1) / kReduceOut;
    if (grid > (int64_t)a.num_sms * 8) grid = (int64_t)a.num_sms * 8;
    bwd_reduce_kernel<<<(unsigned)grid, kReduceThreads, 0, a.stream>>>(part, a.B, a.Skv, a.D, pl.Dp, pl.U, tab,
                                                           pl.nchunks, pl.CH, pl.QT, pl.qtiles, a.ratio,
                                                           a.ks == nullptr ? 1 : 0, a.grad_dtype, a.dk);
    return cudaGetLastError();
}

}  // namespace lidx
