// gather.cu -- the V4 forward with precomputed top-k indices ("tilelang_indexer"
// page, V4IndexerFunction.forward / v4_lighting_indexer: optional
// topk_indices [batch, seqlen, topk] int32): no selection; the score of each
// given (row, key) pair is computed directly, without a dense sweep:
//     score[b,s,j] = sum_h w[s,b,h] * act(q[s,b,h,:] . k[t,b,:]),  t = idx[b,s,j],
// and -inf where t lies outside the row's causal range [0, min((s+1)/ratio, Skv)).
//
// One CTA per query row; the given keys are gathered in chunks of 64 and
// x = Q . Kc^T runs on warp-level tf32 MMA tiles (q and k are exact in tf32,
// accumulation fp32); the weighted head sum is reduced across lanes and warps.
// H below 16 uses plain FMA loops.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lidx {

constexpr int kGatThreads = 256;
constexpr int kGatJ = 64;

__device__ __forceinline__ float gat_bf16(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

template <int H>
__global__ void __launch_bounds__(kGatThreads)
    gather_scores_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                         const float* __restrict__ w, const int32_t* __restrict__ idx, int B, int S,
                         int Skv, int D, int ratio, int topk, int act, int32_t* __restrict__ out_idx,
                         float* __restrict__ out_sc) {
    extern __shared__ __align__(16) float sm[];
    const int DP = D + 4;
    float* qs = sm;                    // [H][DP]
    float* kc = qs + H * DP;           // [J][DP]
    float* ws = kc + kGatJ * DP;       // [H]
    float* colsum = ws + H;            // [J]
    int* ts = reinterpret_cast<int*>(colsum + kGatJ);  // [J]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c4 = lane & 3;
    constexpr int NWARP = kGatThreads / 32;
    const float ninf = __int_as_float(0xff800000);
    auto u32 = [](float x) { return __float_as_uint(x); };

    for (int r = blockIdx.x; r < B * S; r += gridDim.x) {
        const int b = r / S, s = r % S;
        const long long ke_ll = (long long)(s + 1) / ratio;
        const int ke = (int)(ke_ll < Skv ? ke_ll : Skv);
        __syncthreads();
        for (int e = tid; e < H * D; e += kGatThreads) {
            const int h = e / D, d = e % D;
            qs[h * DP + d] = gat_bf16(q[(((size_t)s * B + b) * H + h) * D + d]);
        }
        for (int h = tid; h < H; h += kGatThreads) ws[h] = w[((size_t)s * B + b) * H + h];
        const int32_t* irow = idx + (size_t)r * topk;
        for (int j0 = 0; j0 < topk; j0 += kGatJ) {
            __syncthreads();
            for (int j = tid; j < kGatJ; j += kGatThreads) {
                const int slot = j0 + j;
                int t = slot < topk ? irow[slot] : -1;
                if (slot < topk) out_idx[(size_t)r * topk + slot] = t;  // copied through
                if (t < 0 || t >= ke) t = -1;
                ts[j] = t;
                colsum[j] = 0.f;
            }
            __syncthreads();
            for (int e = tid; e < kGatJ * D; e += kGatThreads) {
                const int j = e / D, d = e % D;
                const int t = ts[j];
                kc[j * DP + d] = t >= 0 ? gat_bf16(k[((size_t)t * B + b) * D + d]) : 0.f;
            }
            __syncthreads();
            if constexpr (H % 16 == 0) {
                constexpr int MT = H / 16;
                for (int tt = warp; tt < MT * (kGatJ / 8); tt += NWARP) {
                    const int mt = tt / (kGatJ / 8), nt = tt % (kGatJ / 8);
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
                    const float* qa = qs + (mt * 16 + g) * DP + c4;
                    const float* kb = kc + (nt * 8 + g) * DP + c4;
                    for (int kk = 0; kk < D; kk += 8)
                        mma_tf32(x, u32(qa[kk]), u32(qa[8 * DP + kk]), u32(qa[kk + 4]),
                                 u32(qa[8 * DP + kk + 4]), u32(kb[kk]), u32(kb[kk + 4]));
                    // weighted head terms of columns 2*c4 and 2*c4+1; sum over this tile's 16 heads
                    float p0 = 0.f, p1 = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = mt * 16 + g + (e >> 1) * 8;
                        const float a = act == 0 ? fmaxf(x[e], 0.f) : x[e];
                        if (e & 1) p1 = fmaf(ws[h], a, p1); else p0 = fmaf(ws[h], a, p0);
                    }
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        p0 += __shfl_xor_sync(0xffffffffu, p0, o);
                        p1 += __shfl_xor_sync(0xffffffffu, p1, o);
                    }
                    if (g == 0) {
                        atomicAdd(&colsum[nt * 8 + 2 * c4], p0);
                        atomicAdd(&colsum[nt * 8 + 2 * c4 + 1], p1);
                    }
                }
            } else {
                for (int e = tid; e < H * kGatJ; e += kGatThreads) {
                    const int h = e / kGatJ, j = e % kGatJ;
                    float x = 0.f;
                    for (int d = 0; d < D; ++d) x = fmaf(qs[h * DP + d], kc[j * DP + d], x);
                    atomicAdd(&colsum[j], ws[h] * (act == 0 ? fmaxf(x, 0.f) : x));
                }
            }
            __syncthreads();
            for (int j = tid; j < kGatJ; j += kGatThreads) {
                const int slot = j0 + j;
                if (slot < topk) out_sc[(size_t)r * topk + slot] = ts[j] >= 0 ? colsum[j] : ninf;
            }
        }
    }
}

template <int H>
static cudaError_t gather_h(const GatherLaunch& a) {
    const int DP = a.D + 4;
    const size_t smem = sizeof(float) * ((size_t)H * DP + (size_t)kGatJ * DP + H + kGatJ) + sizeof(int) * kGatJ;
    auto kern = gather_scores_kernel<H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGatThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)a.num_sms * per_sm;
    const int64_t rows = (int64_t)a.B * a.S;
    if (grid > rows) grid = rows;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, kGatThreads, smem, a.stream>>>((const uint16_t*)a.q, (const uint16_t*)a.k, a.w,
                                                         a.idx, a.B, a.S, a.Skv, a.D, a.ratio, a.topk, a.act,
                                                         a.out_idx, a.out_sc);
    return cudaGetLastError();
}

cudaError_t gather_launch(const GatherLaunch& a) {
    switch (a.H) {
        case 1: return gather_h<1>(a);
        case 2: return gather_h<2>(a);
        case 4: return gather_h<4>(a);
        case 8: return gather_h<8>(a);
        case 16: return gather_h<16>(a);
        case 32: return gather_h<32>(a);
        case 64: return gather_h<64>(a);
        case 128: return gather_h<128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lidx
