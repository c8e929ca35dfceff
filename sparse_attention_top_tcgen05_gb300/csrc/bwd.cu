// bwd.cu -- backward of the V4 indexer through the selected entries
// ("tilelang_indexer" page, V4IndexerFunction.backward(grad_scores,
// grad_indices); grad_indices carries no gradient).
//
// For query row (b,s) and selected slot j with key t = idx[j] inside the row's
// causal range and g = grad[j], with x_h = q[s,b,h,:] . k[t,b,:]:
//     dw[s,b,h]   += g * act(x_h)
//     c_h          = g * w[s,b,h] * act'(x_h)          (ReLU'(0) = 0)
//     dq[s,b,h,:] += c_h * k[t,b,:]
//     dk[t,b,:]   += sum_h c_h * q[s,b,h,:]
//
// One CTA per query row.  The row's queries stay in shared memory; its
// selected keys are gathered in chunks of J.  Per chunk three small
// contractions run, on warp-level tf32 MMA tiles when H is a multiple of 16
// (bwd_rows_mma_kernel) and on the CUDA cores with register tiles of four
// otherwise (bwd_rows_kernel):
//     X [H x J]  = Q [H x D] . Kc^T        (then dw and C = g*w*act'(x))
//     dq[H x D] += C [H x J] . Kc [J x D]  (accumulated in registers)
//     dKc[J x D] = C^T [J x H] . Q [H x D] (scatter-added to dk)
// dq and dw are written once per row; dk is cleared by the caller-side
// launcher and accumulated with atomics (order-dependent in the last bits).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lidx {

constexpr int kBwdThreads = 256;
constexpr int kBwdJ = 64;  // selected keys per chunk

__device__ __forceinline__ float bf16_to_f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

template <int H>
__global__ void __launch_bounds__(kBwdThreads)
    bwd_rows_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                    const float* __restrict__ w, const int32_t* __restrict__ idx,
                    const float* __restrict__ grad, int B, int S, int Skv, int D, int ratio,
                    const int32_t* __restrict__ ksa, const int32_t* __restrict__ kea,
                    int topk, int act, float* __restrict__ dq, float* __restrict__ dk,
                    float* __restrict__ dw) {
    extern __shared__ __align__(16) float sm[];
    const int DP = D + 4;                      // padded row stride (keeps 16-byte alignment)
    float* qs = sm;                            // [H][DP]
    float* kc = qs + H * DP;                   // [J][DP]   gathered keys
    float* kT = kc + kBwdJ * DP;               // [D][J+4]  the same keys transposed
    float* cs = kT + D * (kBwdJ + 4);          // [H][J+4]  C = g*w*act'(x)
    float* ws = cs + H * (kBwdJ + 4);          // [H]
    float* dws = ws + H;                       // [H]
    float* gs = dws + H;                       // [J]
    int* ts = reinterpret_cast<int*>(gs + kBwdJ);  // [J]   key, or -1
    const int tid = threadIdx.x;
    const int D4 = D / 4;
    constexpr int JP = kBwdJ + 4;
    // fixed work split of the three contractions
    const int nX = H * (kBwdJ / 4);            // groups (h, 4 keys)
    const int nQ = H * D4;                     // groups (h, 4 dims)
    const int nK = kBwdJ * D4;                 // groups (key, 4 dims)
    constexpr int MAXQ = (H * 32 + kBwdThreads - 1) / kBwdThreads;  // D <= 128

    for (int r = blockIdx.x; r < B * S; r += gridDim.x) {
        const int b = r / S, s = r % S;
        int ks = 0, ke;
        if (ksa) {
            ks = ksa[s] > 0 ? ksa[s] : 0;
            ke = kea[s] < Skv ? kea[s] : Skv;
        } else {
            const long long ke_ll = (long long)(s + 1) / ratio;
            ke = (int)(ke_ll < Skv ? ke_ll : Skv);
        }
        __syncthreads();  // previous row done with shared memory
        for (int e = tid; e < H * D; e += kBwdThreads) {
            const int h = e / D, d = e % D;
            qs[h * DP + d] = bf16_to_f(q[(((size_t)s * B + b) * H + h) * D + d]);
        }
        for (int h = tid; h < H; h += kBwdThreads) {
            ws[h] = w[((size_t)s * B + b) * H + h];
            dws[h] = 0.f;
        }
        float accq[MAXQ][4];
#pragma unroll
        for (int i = 0; i < MAXQ; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) accq[i][c] = 0.f;

        const int32_t* irow = idx + (size_t)r * topk;
        const float* grow = grad + (size_t)r * topk;
        for (int j0 = 0; j0 < topk; j0 += kBwdJ) {
            __syncthreads();  // previous chunk done with kc/kT/cs
            for (int j = tid; j < kBwdJ; j += kBwdThreads) {
                const int slot = j0 + j;
                int t = slot < topk ? irow[slot] : -1;
                if (t < ks || t >= ke) t = -1;  // padding or outside the causal range
                ts[j] = t;
                gs[j] = t >= 0 ? grow[slot] : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < kBwdJ * D; e += kBwdThreads) {
                const int j = e / D, d = e % D;
                const int t = ts[j];
                const float v = t >= 0 ? bf16_to_f(k[((size_t)t * B + b) * D + d]) : 0.f;
                kc[j * DP + d] = v;
                kT[d * JP + j] = v;
            }
            __syncthreads();
            // X and C: thread group (h, four keys)
            for (int gi = tid; gi < nX; gi += kBwdThreads) {
                const int h = gi / (kBwdJ / 4), j4 = (gi % (kBwdJ / 4)) * 4;
                float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                const float* qh = qs + h * DP;
                for (int d = 0; d < D; ++d) {
                    const float qv = qh[d];
                    const float4 kv = *reinterpret_cast<const float4*>(kT + d * JP + j4);
                    x0 = fmaf(qv, kv.x, x0);
                    x1 = fmaf(qv, kv.y, x1);
                    x2 = fmaf(qv, kv.z, x2);
                    x3 = fmaf(qv, kv.w, x3);
                }
                const float xs[4] = {x0, x1, x2, x3};
                float dwp = 0.f, cv[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float g = gs[j4 + c];
                    const float x = xs[c];
                    const float a = act == 0 ? fmaxf(x, 0.f) : x;
                    const float da = act == 0 ? (x > 0.f ? 1.f : 0.f) : 1.f;
                    dwp = fmaf(g, a, dwp);
                    cv[c] = g * ws[h] * da;
                }
                *reinterpret_cast<float4*>(cs + h * JP + j4) = make_float4(cv[0], cv[1], cv[2], cv[3]);
                atomicAdd(&dws[h], dwp);
            }
            __syncthreads();
            // dq += C . Kc: thread group (h, four dims), kept in registers across chunks
#pragma unroll
            for (int i = 0; i < MAXQ; ++i) {
                const int gi = tid + i * kBwdThreads;
                if (gi < nQ) {
                    const int h = gi / D4, d4 = (gi % D4) * 4;
                    const float* ch = cs + h * JP;
                    float a0 = accq[i][0], a1 = accq[i][1], a2 = accq[i][2], a3 = accq[i][3];
                    for (int j = 0; j < kBwdJ; ++j) {
                        const float cvj = ch[j];
                        const float4 kv = *reinterpret_cast<const float4*>(kc + j * DP + d4);
                        a0 = fmaf(cvj, kv.x, a0);
                        a1 = fmaf(cvj, kv.y, a1);
                        a2 = fmaf(cvj, kv.z, a2);
                        a3 = fmaf(cvj, kv.w, a3);
                    }
                    accq[i][0] = a0;
                    accq[i][1] = a1;
                    accq[i][2] = a2;
                    accq[i][3] = a3;
                }
            }
            // dk[t] += C^T . Q: thread group (key, four dims)
            for (int gi = tid; gi < nK; gi += kBwdThreads) {
                const int j = gi / D4, d4 = (gi % D4) * 4;
                const int t = ts[j];
                if (t < 0) continue;
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                for (int h = 0; h < H; ++h) {
                    const float cvh = cs[h * JP + j];
                    const float4 qv = *reinterpret_cast<const float4*>(qs + h * DP + d4);
                    a0 = fmaf(cvh, qv.x, a0);
                    a1 = fmaf(cvh, qv.y, a1);
                    a2 = fmaf(cvh, qv.z, a2);
                    a3 = fmaf(cvh, qv.w, a3);
                }
                float* o = dk + ((size_t)t * B + b) * D + d4;
                atomicAdd(o + 0, a0);
                atomicAdd(o + 1, a1);
                atomicAdd(o + 2, a2);
                atomicAdd(o + 3, a3);
            }
        }
        // dq and dw of this row
#pragma unroll
        for (int i = 0; i < MAXQ; ++i) {
            const int gi = tid + i * kBwdThreads;
            if (gi < nQ) {
                const int h = gi / D4, d4 = (gi % D4) * 4;
                *reinterpret_cast<float4*>(dq + (((size_t)s * B + b) * H + h) * D + d4) =
                    make_float4(accq[i][0], accq[i][1], accq[i][2], accq[i][3]);
            }
        }
        __syncthreads();
        for (int h = tid; h < H; h += kBwdThreads) dw[((size_t)s * B + b) * H + h] = dws[h];
    }
}

// Same computation as bwd_rows_kernel with the three contractions on warp-level
// tf32 MMA tiles (m16n8k8).  q and k are exact in tf32 (bf16 values); the
// accumulators are fp32; C = g*w*act'(x) is rounded to tf32 (nearest).  Fragment
// coordinates: g = lane/4, c = lane%4; A rows g and g+8, columns c and c+4;
// B column g, rows c and c+4; D rows g and g+8, columns 2c and 2c+1.
template <int H>
__global__ void __launch_bounds__(kBwdThreads)
    bwd_rows_mma_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                        const float* __restrict__ w, const int32_t* __restrict__ idx,
                        const float* __restrict__ grad, int B, int S, int Skv, int D, int ratio,
                        const int32_t* __restrict__ ksa, const int32_t* __restrict__ kea,
                        int topk, int act, float* __restrict__ dq, float* __restrict__ dk,
                        float* __restrict__ dw) {
    static_assert(H % 16 == 0, "H must be a multiple of 16");
    extern __shared__ __align__(16) float sm[];
    const int DP = D + 4;
    constexpr int JP = kBwdJ + 4;
    float* qs = sm;                      // [H][DP]
    float* kc = qs + H * DP;             // [J][DP]
    float* cs = kc + kBwdJ * DP;         // [H][JP]  C as tf32
    float* ws = cs + H * JP;             // [H]
    float* dws = ws + H;                 // [H]
    float* gs = dws + H;                 // [J]
    int* ts = reinterpret_cast<int*>(gs + kBwdJ);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c4 = lane & 3;
    constexpr int NWARP = kBwdThreads / 32;
    constexpr int MT = H / 16;
    const int NTD = D / 8;
    constexpr int QT_MAX = (MT * 16 + NWARP - 1) / NWARP;  // dq tiles per warp at D = 128
    auto u32 = [](float x) { return __float_as_uint(x); };

    for (int r = blockIdx.x; r < B * S; r += gridDim.x) {
        const int b = r / S, s = r % S;
        int ks = 0, ke;
        if (ksa) {
            ks = ksa[s] > 0 ? ksa[s] : 0;
            ke = kea[s] < Skv ? kea[s] : Skv;
        } else {
            const long long ke_ll = (long long)(s + 1) / ratio;
            ke = (int)(ke_ll < Skv ? ke_ll : Skv);
        }
        __syncthreads();
        for (int e = tid; e < H * D; e += kBwdThreads) {
            const int h = e / D, d = e % D;
            qs[h * DP + d] = bf16_to_f(q[(((size_t)s * B + b) * H + h) * D + d]);
        }
        for (int h = tid; h < H; h += kBwdThreads) {
            ws[h] = w[((size_t)s * B + b) * H + h];
            dws[h] = 0.f;
        }
        float accq[QT_MAX][4];
#pragma unroll
        for (int i = 0; i < QT_MAX; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) accq[i][e] = 0.f;

        const int32_t* irow = idx + (size_t)r * topk;
        const float* grow = grad + (size_t)r * topk;
        for (int j0 = 0; j0 < topk; j0 += kBwdJ) {
            __syncthreads();
            for (int j = tid; j < kBwdJ; j += kBwdThreads) {
                const int slot = j0 + j;
                int t = slot < topk ? irow[slot] : -1;
                if (t < ks || t >= ke) t = -1;
                ts[j] = t;
                gs[j] = t >= 0 ? grow[slot] : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < kBwdJ * D; e += kBwdThreads) {
                const int j = e / D, d = e % D;
                const int t = ts[j];
                kc[j * DP + d] = t >= 0 ? bf16_to_f(k[((size_t)t * B + b) * D + d]) : 0.f;
            }
            __syncthreads();
            // X = Q . Kc^T  [H x J]; then C and dw
            for (int tt = warp; tt < MT * (kBwdJ / 8); tt += NWARP) {
                const int mt = tt / (kBwdJ / 8), nt = tt % (kBwdJ / 8);
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                const float* qa = qs + (mt * 16 + g) * DP + c4;
                const float* kb = kc + (nt * 8 + g) * DP + c4;
                for (int kk = 0; kk < D; kk += 8)
                    mma_tf32(x, u32(qa[kk]), u32(qa[8 * DP + kk]), u32(qa[kk + 4]), u32(qa[8 * DP + kk + 4]),
                             u32(kb[kk]), u32(kb[kk + 4]));
                float dwp[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = mt * 16 + g + (e >> 1) * 8, j = nt * 8 + 2 * c4 + (e & 1);
                    const float xv = x[e], gv = gs[j];
                    const float a = act == 0 ? fmaxf(xv, 0.f) : xv;
                    const float da = act == 0 ? (xv > 0.f ? 1.f : 0.f) : 1.f;
                    dwp[e >> 1] = fmaf(gv, a, dwp[e >> 1]);
                    cs[h * JP + j] = __uint_as_float(tf32_round(gv * ws[h] * da));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    dwp[u] += __shfl_xor_sync(0xffffffffu, dwp[u], 1);
                    dwp[u] += __shfl_xor_sync(0xffffffffu, dwp[u], 2);
                }
                if (c4 == 0) {
                    atomicAdd(&dws[mt * 16 + g], dwp[0]);
                    atomicAdd(&dws[mt * 16 + g + 8], dwp[1]);
                }
            }
            __syncthreads();
            // dq += C . Kc  [H x D], tiles kept in registers across chunks
#pragma unroll
            for (int i = 0; i < QT_MAX; ++i) {
                const int tt = warp + i * NWARP;
                if (tt < MT * NTD) {
                    const int mt = tt / NTD, nt = tt % NTD;
                    const float* ca = cs + (mt * 16 + g) * JP + c4;
                    const float* kb = kc + c4 * DP + nt * 8 + g;
#pragma unroll
                    for (int kk = 0; kk < kBwdJ; kk += 8)
                        mma_tf32(accq[i], u32(ca[kk]), u32(ca[8 * JP + kk]), u32(ca[kk + 4]),
                                 u32(ca[8 * JP + kk + 4]), u32(kb[kk * DP]), u32(kb[(kk + 4) * DP]));
                }
            }
            // dKc = C^T . Q  [J x D], scatter-added to dk
            for (int tt = warp; tt < (kBwdJ / 16) * NTD; tt += NWARP) {
                const int mt = tt / NTD, nt = tt % NTD;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                const float* ca = cs + c4 * JP + mt * 16 + g;  // A[j][h] = C[h][j]
                const float* qb = qs + c4 * DP + nt * 8 + g;
#pragma unroll
                for (int kk = 0; kk < H; kk += 8)
                    mma_tf32(acc, u32(ca[kk * JP]), u32(ca[kk * JP + 8]), u32(ca[(kk + 4) * JP]),
                             u32(ca[(kk + 4) * JP + 8]), u32(qb[kk * DP]), u32(qb[(kk + 4) * DP]));
                // Lanes c4 and c4^1 swap halves so that each holds four consecutive d of
                // one key (even c4: key row g, odd c4: key row g + 8), then one 16-byte
                // vector reduction per lane instead of four scalar ones.
                const bool odd = (c4 & 1) != 0;
                const float s0 = __shfl_xor_sync(0xffffffffu, odd ? acc[0] : acc[2], 1);
                const float s1 = __shfl_xor_sync(0xffffffffu, odd ? acc[1] : acc[3], 1);
                const int j = mt * 16 + g + (odd ? 8 : 0);
                const int d0 = nt * 8 + 2 * (c4 & 2);
                const int t = ts[j];
                if (t >= 0) {
                    const float4 v = odd ? make_float4(s0, s1, acc[2], acc[3])
                                         : make_float4(acc[0], acc[1], s0, s1);
                    atomicAdd(reinterpret_cast<float4*>(dk + ((size_t)t * B + b) * D + d0), v);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < QT_MAX; ++i) {
            const int tt = warp + i * NWARP;
            if (tt < MT * NTD) {
                const int mt = tt / NTD, nt = tt % NTD;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = mt * 16 + g + (e >> 1) * 8, d = nt * 8 + 2 * c4 + (e & 1);
                    dq[(((size_t)s * B + b) * H + h) * D + d] = accq[i][e];
                }
            }
        }
        __syncthreads();
        for (int h = tid; h < H; h += kBwdThreads) dw[((size_t)s * B + b) * H + h] = dws[h];
    }
}

static size_t bwd_mma_smem(int H, int D) {
    const int DP = D + 4, JP = kBwdJ + 4;
    return sizeof(float) * ((size_t)H * DP + (size_t)kBwdJ * DP + (size_t)H * JP + 2 * (size_t)H + kBwdJ) +
           sizeof(int) * kBwdJ;
}

template <int H>
static cudaError_t bwd_mma_h(const BwdLaunch& a) {
    const size_t smem = bwd_mma_smem(H, a.D);
    auto kern = bwd_rows_mma_kernel<H>;
    cudaError_t e = set_smem_attr((const void*)kern, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBwdThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)a.num_sms * per_sm;
    const int64_t rows = (int64_t)a.B * a.S;
    if (grid > rows) grid = rows;
    kern<<<(unsigned)grid, kBwdThreads, smem, a.stream>>>(
        (const uint16_t*)a.q, (const uint16_t*)a.k, a.w, a.idx, a.grad, a.B, a.S, a.Skv, a.D, a.ratio,
        a.ks, a.ke, a.topk, a.act, (float*)a.dq, (float*)a.dk, a.dw);
    return cudaGetLastError();
}

static size_t bwd_smem(int H, int D) {
    const int DP = D + 4, JP = kBwdJ + 4;
    return sizeof(float) * ((size_t)H * DP + (size_t)kBwdJ * DP + (size_t)D * JP + (size_t)H * JP +
                            2 * (size_t)H + kBwdJ) +
           sizeof(int) * kBwdJ;
}

template <int H>
static cudaError_t bwd_h(const BwdLaunch& a) {
    const size_t smem = bwd_smem(H, a.D);
    auto kern = bwd_rows_kernel<H>;
    cudaError_t e = set_smem_attr((const void*)kern, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBwdThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)a.num_sms * per_sm;
    const int64_t rows = (int64_t)a.B * a.S;
    if (grid > rows) grid = rows;
    kern<<<(unsigned)grid, kBwdThreads, smem, a.stream>>>(
        (const uint16_t*)a.q, (const uint16_t*)a.k, a.w, a.idx, a.grad, a.B, a.S, a.Skv, a.D, a.ratio,
        a.ks, a.ke, a.topk, a.act, (float*)a.dq, (float*)a.dk, a.dw);
    return cudaGetLastError();
}

LIDX_STATUS_READER(status_bwd)

size_t bwd_workspace_bytes(int64_t, int64_t, int64_t, int, int, int, int) { return 0; }

cudaError_t bwd_launch(const BwdLaunch& a) {
    // dk is a sum over rows: clear it first (dq and dw are written whole)
    cudaError_t e = cudaMemsetAsync(a.dk, 0, sizeof(float) * (size_t)a.Skv * a.B * a.D, a.stream);
    if (e != cudaSuccess) return e;
    if ((int64_t)a.B * a.S == 0) return cudaSuccess;
    switch (a.H) {
        case 1: return bwd_h<1>(a);
        case 2: return bwd_h<2>(a);
        case 4: return bwd_h<4>(a);
        case 8: return bwd_h<8>(a);
        case 16: return bwd_mma_h<16>(a);
        case 32: return bwd_mma_h<32>(a);
        case 64: return bwd_mma_h<64>(a);
        case 128: return bwd_mma_h<128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lidx
