// v41.cu -- visibility pass of the V4.1 scorer ("deepseek_v41.indexer" page,
// indexer_scores: boolean `allowed` [batch, local_sequence, global_compressed]).
//
// One streaming read of `allowed` decides, for every (query tile, 128-key tile)
// block, whether any pair in it is visible.  Blocks with no visible pair get
// their scores written here as -inf, so the tensor-core pass touches only
// blocks with work and every output element is written exactly once.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lidx {

constexpr int kMaskThreads = 256;

// Grid-stride over (b, query tile); each warp takes key tiles in turn.  Lane l
// covers keys [kt*128 + 4l, kt*128 + 4l + 4) of every row of the tile.
__global__ void __launch_bounds__(kMaskThreads)
    v41_mask_kernel(const uint8_t* __restrict__ allowed, uint16_t* __restrict__ out,
                    uint8_t* __restrict__ tilemap, int B, int S, int Skv, int QT, int qtiles,
                    int ntk) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = kMaskThreads / 32;
    const bool vec = (Skv & 3) == 0;  // rows start 4-byte aligned: word loads, 8-byte stores
    const int units = B * qtiles;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int b = unit / qtiles, qt = unit % qtiles, s0 = qt * QT;
        const int rows = min(QT, S - s0);
        for (int kt = warp; kt < ntk; kt += NW) {
            const int t0 = kt * 128 + lane * 4;
            uint32_t any = 0;
            for (int r = 0; r < rows; ++r) {
                const uint8_t* row = allowed + ((size_t)b * S + s0 + r) * Skv;
                if (vec && t0 + 3 < Skv) {
                    any |= *reinterpret_cast<const uint32_t*>(row + t0);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (t0 + j < Skv) any |= row[t0 + j];
                }
            }
            const bool active = __any_sync(0xffffffffu, any != 0);
            if (lane == 0) tilemap[(size_t)unit * ntk + kt] = active ? 1 : 0;
            if (!active) {
                for (int r = 0; r < rows; ++r) {
                    uint16_t* o = out + ((size_t)b * S + s0 + r) * Skv;
                    if (vec && t0 + 3 < Skv) {
                        *reinterpret_cast<uint2*>(o + t0) = make_uint2(0xFF80FF80u, 0xFF80FF80u);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (t0 + j < Skv) o[t0 + j] = 0xFF80u;
                    }
                }
            }
        }
    }
}

// Same pass for 16-byte aligned rows (Skv % 16 == 0, aligned bases): each lane
// reads 16 flags of up to four rows at once, so a warp keeps 2 KB of `allowed`
// in flight and covers four key tiles (8 lanes each) per step.
__global__ void __launch_bounds__(kMaskThreads)
    v41_mask_kernel16(const uint8_t* __restrict__ allowed, uint16_t* __restrict__ out,
                      uint8_t* __restrict__ tilemap, int B, int S, int Skv, int QT, int qtiles,
                      int ntk) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = kMaskThreads / 32;
    const int units = B * qtiles;
    const int nchunks = (ntk + 3) / 4;  // 512-key chunks
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int b = unit / qtiles, qt = unit % qtiles, s0 = qt * QT;
        const int rows = min(QT, S - s0);
        for (int ch = warp; ch < nchunks; ch += NW) {
            const int t0 = ch * 512 + lane * 16;
            const bool in = t0 < Skv;  // Skv % 16 == 0: all 16 keys inside or none
            const uint8_t* base = allowed + ((size_t)b * S + s0) * Skv + (in ? t0 : 0);
            uint32_t acc = 0;
            int r = 0;
            for (; r + 4 <= rows; r += 4) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[u] = in ? *reinterpret_cast<const uint4*>(base + (size_t)(r + u) * Skv)
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) acc |= v[u].x | v[u].y | v[u].z | v[u].w;
            }
            for (; r < rows; ++r) {
                const uint4 v = in ? *reinterpret_cast<const uint4*>(base + (size_t)r * Skv)
                                   : make_uint4(0u, 0u, 0u, 0u);
                acc |= v.x | v.y | v.z | v.w;
            }
            // any visible pair in this lane's 128-key tile (lanes 8g .. 8g+7)
            uint32_t any = acc != 0 ? 1u : 0u;
            any |= __shfl_xor_sync(0xffffffffu, any, 1);
            any |= __shfl_xor_sync(0xffffffffu, any, 2);
            any |= __shfl_xor_sync(0xffffffffu, any, 4);
            const int kt = ch * 4 + (lane >> 3);
            if ((lane & 7) == 0 && kt < ntk) tilemap[(size_t)unit * ntk + kt] = any ? 1 : 0;
            if (!any && in) {
                const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
                uint16_t* o = out + ((size_t)b * S + s0) * Skv + t0;
                for (int r2 = 0; r2 < rows; ++r2) {
                    uint4* d = reinterpret_cast<uint4*>(o + (size_t)r2 * Skv);
                    d[0] = ninf;
                    d[1] = ninf;
                }
            }
        }
    }
}

cudaError_t v41_mask_launch(const uint8_t* allowed, uint16_t* out, uint8_t* tilemap, int B, int S,
                            int Skv, int QT, cudaStream_t stream) {
    const int qtiles = (S + QT - 1) / QT, ntk = (Skv + 127) / 128;
    const int64_t units = (int64_t)B * qtiles;
    if (units == 0 || ntk == 0) return cudaSuccess;
    const int sms = current_sms();
    int64_t grid = (int64_t)sms * 8;
    if (grid > units) grid = units;
    if ((Skv & 15) == 0 && ((((uintptr_t)allowed) | ((uintptr_t)out)) & 15) == 0)
        v41_mask_kernel16<<<(unsigned)grid, kMaskThreads, 0, stream>>>(allowed, out, tilemap, B, S,
                                                                       Skv, QT, qtiles, ntk);
    else
        v41_mask_kernel<<<(unsigned)grid, kMaskThreads, 0, stream>>>(allowed, out, tilemap, B, S, Skv,
                                                                     QT, qtiles, ntk);
    return cudaGetLastError();
}

}  // namespace lidx
