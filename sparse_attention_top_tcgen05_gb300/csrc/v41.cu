// v41.cu -- visibility pass of the V4.1 scorer ("deepseek_v41.indexer" page,
// indexer_scores: boolean `allowed` [batch, local_sequence, global_compressed]).
//
// One streaming read of `allowed` decides, for every (query tile, 128-key tile)
// block, whether any pair in it is visible, and for every query tile the range
// of key tiles that holds its visible pairs.  The scoring kernel then computes
// the blocks with a visible pair and writes -inf over the others.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace lidx {

constexpr int kMaskThreads = 256;

// The unit's record: key tiles [first, last] hold every visible pair, and bit j
// of the 64-bit mask is the tile map's entry for key tile first + j (one warp;
// the map row was written by this block before the caller's barrier).
__device__ __forceinline__ void write_unit_record(const uint8_t* map, int first, int last, int lane,
                                                  int4* rec) {
    int4 r = make_int4(0, 0, 0, 0);
    if (last >= 0) {
        const int j0 = first + lane, j1 = first + 32 + lane;
        const uint32_t m0 = __ballot_sync(0xffffffffu, j0 <= last && map[j0] != 0);
        const uint32_t m1 = __ballot_sync(0xffffffffu, j1 <= last && map[j1] != 0);
        r = make_int4(first, last + 1, (int)m0, (int)m1);
    }
    if (lane == 0) *rec = r;
}

// Grid-stride over (b, query tile); each warp takes key tiles in turn.  Lane l
// covers keys [kt*128 + 4l, kt*128 + 4l + 4) of every row of the tile.
__global__ void __launch_bounds__(kMaskThreads)
    v41_mask_kernel(const uint8_t* __restrict__ allowed, uint8_t* __restrict__ tilemap, int4* __restrict__ urec, int B, int S, int Skv,
                    int QT, int qtiles, int ntk) {
    __shared__ int s_first, s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();  // the scoring kernel may start its set-up now
    constexpr int NW = kMaskThreads / 32;
    const bool vec = (Skv & 3) == 0;  // rows start 4-byte aligned: word loads
    const int units = B * qtiles;
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int b = unit / qtiles, qt = unit % qtiles, s0 = qt * QT;
        const int rows = min(QT, S - s0);
        __syncthreads();  // the previous unit's range is written out
        if (threadIdx.x == 0) {
            s_first = ntk;
            s_last = -1;
        }
        __syncthreads();
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
            if (lane == 0) {
                tilemap[(size_t)unit * ntk + kt] = active ? 1 : 0;
                if (active) {
                    atomicMin(&s_first, kt);
                    atomicMax(&s_last, kt);
                }
            }
        }
        __syncthreads();
        if (warp == 0) write_unit_record(tilemap + (size_t)unit * ntk, s_first, s_last, lane, urec + unit);
    }
}

// Same pass for 16-byte aligned rows (Skv % 16 == 0, aligned bases): each lane
// reads 16 flags of up to four rows at once, so a warp keeps 2 KB of `allowed`
// in flight and covers four key tiles (8 lanes each) per step.
__global__ void __launch_bounds__(kMaskThreads)
    v41_mask_kernel16(const uint8_t* __restrict__ allowed, uint8_t* __restrict__ tilemap, int4* __restrict__ urec, int B, int S,
                      int Skv, int QT, int qtiles, int ntk) {
    __shared__ int s_first, s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();  // the scoring kernel may start its set-up now
    constexpr int NW = kMaskThreads / 32;
    const int units = B * qtiles;
    const int nchunks = (ntk + 3) / 4;  // 512-key chunks
    for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int b = unit / qtiles, qt = unit % qtiles, s0 = qt * QT;
        const int rows = min(QT, S - s0);
        __syncthreads();  // the previous unit's range is written out
        if (threadIdx.x == 0) {
            s_first = ntk;
            s_last = -1;
        }
        __syncthreads();
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
            if ((lane & 7) == 0 && kt < ntk) {
                tilemap[(size_t)unit * ntk + kt] = any ? 1 : 0;
                if (any) {
                    atomicMin(&s_first, kt);
                    atomicMax(&s_last, kt);
                }
            }
        }
        __syncthreads();
        if (warp == 0) write_unit_record(tilemap + (size_t)unit * ntk, s_first, s_last, lane, urec + unit);
    }
}

cudaError_t v41_mask_launch(const uint8_t* allowed, uint8_t* tilemap, int4* urec, int B, int S, int Skv,
                            int QT, cudaStream_t stream) {
    const int qtiles = (S + QT - 1) / QT, ntk = (Skv + 127) / 128;
    const int64_t units = (int64_t)B * qtiles;
    if (units == 0 || ntk == 0) return cudaSuccess;
    const int sms = current_sms();
    int64_t grid = (int64_t)sms * 8;
    if (grid > units) grid = units;
    if ((Skv & 15) == 0 && (((uintptr_t)allowed) & 15) == 0)
        v41_mask_kernel16<<<(unsigned)grid, kMaskThreads, 0, stream>>>(allowed, tilemap, urec, B, S, Skv,
                                                                       QT, qtiles, ntk);
    else
        v41_mask_kernel<<<(unsigned)grid, kMaskThreads, 0, stream>>>(allowed, tilemap, urec, B, S, Skv, QT,
                                                                     qtiles, ntk);
    return cudaGetLastError();
}

}  // namespace lidx
