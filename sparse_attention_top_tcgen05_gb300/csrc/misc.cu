// misc.cu -- small memory-bound kernels: gather of scores at given indices
// ("tilelang_indexer" page, pytorch_extract_topk_scores(logits, topk_indices)).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace lidx {

// One thread per output element; consecutive threads read consecutive
// indices (coalesced) and gather from the row's logits (L2-friendly).
__global__ void extract_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                               int64_t rows, int64_t Skv, int topk, float* __restrict__ out) {
    const int64_t n = rows * (int64_t)topk;
    const float ninf = __int_as_float(0xff800000);
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / topk;
        const int32_t t = idx[e];
        out[e] = (t >= 0 && t < Skv) ? logits[r * Skv + t] : ninf;
    }
}

cudaError_t extract_launch(const float* logits, const int32_t* idx, int64_t rows, int64_t Skv,
                           int topk, float* out, cudaStream_t stream) {
    const int64_t n = rows * (int64_t)topk;
    if (n == 0) return cudaSuccess;
    const int sms = current_sms();
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    extract_kernel<<<(unsigned)blocks, 256, 0, stream>>>(logits, idx, rows, Skv, topk, out);
    return cudaGetLastError();
}

// Rows with no visible key: index -1 / score -inf everywhere.
__global__ void pad_kernel(int64_t n, int32_t* __restrict__ idx, float* __restrict__ sc) {
    const float ninf = __int_as_float(0xff800000);
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        idx[e] = -1;
        sc[e] = ninf;
    }
}

cudaError_t pad_launch(int64_t n, int32_t* idx, float* sc, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pad_kernel<<<(unsigned)blocks, 256, 0, stream>>>(n, idx, sc);
    return cudaGetLastError();
}

// The same with bf16 scores (-inf = 0xFF80).
__global__ void pad16_kernel(int64_t n, int32_t* __restrict__ idx, uint16_t* __restrict__ sc) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        idx[e] = -1;
        sc[e] = 0xFF80u;
    }
}

cudaError_t pad16_launch(int64_t n, int32_t* idx, uint16_t* sc, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pad16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(n, idx, sc);
    return cudaGetLastError();
}

// Given indices with no keys to score: indices copied through, scores -inf.
__global__ void copy_pad_kernel(int64_t n, const int32_t* __restrict__ in, int32_t* __restrict__ idx,
                                float* __restrict__ sc) {
    const float ninf = __int_as_float(0xff800000);
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        idx[e] = in[e];
        sc[e] = ninf;
    }
}

cudaError_t copy_pad_launch(int64_t n, const int32_t* in, int32_t* idx, float* sc, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    copy_pad_kernel<<<(unsigned)blocks, 256, 0, stream>>>(n, in, idx, sc);
    return cudaGetLastError();
}

// Standalone selection: each CTA (kTopkRowThreads threads) takes rows in turn.
// Its scratch has a bitmap of 4096 keys, so an all-equal bucket of a row of up
// to 4096 keys is ranked in one chunk.
constexpr int kTopkRowThreads = 256;
using TopkSmemRows = TopkSmemT<kTopkCap, kTopkBuckets, 128>;

__global__ void __launch_bounds__(kTopkRowThreads)
    topk_rows_kernel(const float* __restrict__ logits, int64_t rows, int S, int Skv, int ratio,
                     const int32_t* __restrict__ ks, const int32_t* __restrict__ ke, int topk,
                     int32_t* __restrict__ out_idx, float* __restrict__ out_sc) {
    extern __shared__ uint8_t smem_raw[];
    TopkSmemRows& sm = *reinterpret_cast<TopkSmemRows*>(smem_raw);
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const int s = (int)(r % S);
        int lo, hi;
        if (ks == nullptr) {
            lo = 0;
            const long long e = (long long)(s + 1) / ratio;
            hi = (int)(e < Skv ? e : Skv);
        } else {
            lo = ks[s] > 0 ? ks[s] : 0;
            hi = ke[s] < Skv ? ke[s] : Skv;
            if (hi < lo) hi = lo;
        }
        row_topk<kTopkRowThreads, false, float>(logits + r * (int64_t)Skv, lo, hi, topk,
                                                out_idx + r * topk, out_sc + r * topk, sm,
                                                threadIdx.x, 1);
    }
}

// Top-k of bf16 V4.1 score rows, where -inf marks a key that is not visible:
// candidates are the finite entries.  With `urange`, a row's keys are limited
// to its query tile's range of key tiles, which holds all its visible keys.
// Those spans are short, so a CTA of kTopkBf16Threads threads with a window of
// kTopkBf16Cap members takes each row: more rows are in flight per SM than
// with the full-size scratch, and a longer row takes more windows.
constexpr int kTopkBf16Threads = 128;
constexpr int kTopkBf16Cap = 1024;
constexpr int kTopkBf16Buckets = 384;  // a short span needs fewer buckets to split it
using TopkSmemBf16 = TopkSmemT<kTopkBf16Cap, kTopkBf16Buckets, 128>;

__global__ void __launch_bounds__(kTopkBf16Threads)
    topk_rows_bf16_kernel(const uint16_t* __restrict__ scores, int64_t rows, int S, int Skv,
                          const int2* __restrict__ urange, int QT, int topk, int32_t* __restrict__ out_idx,
                          uint16_t* __restrict__ out_sc) {
    extern __shared__ uint8_t smem_raw[];
    TopkSmemBf16& sm = *reinterpret_cast<TopkSmemBf16*>(smem_raw);
    const int qtiles = (S + QT - 1) / QT;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        int lo = 0, hi = Skv;
        if (urange) {
            const int64_t b = r / S;
            const int s = (int)(r - b * S);
            const int2 kr = urange[b * qtiles + s / QT];
            lo = kr.y > kr.x ? kr.x * 128 : 0;
            hi = kr.y > kr.x ? min(kr.y * 128, Skv) : 0;
        }
        row_topk<kTopkBf16Threads, true, uint16_t>(scores + r * (int64_t)Skv, lo, hi, topk, out_idx + r * topk,
                                                   out_sc + r * topk, sm, threadIdx.x, 1);
    }
}

template <class K>
static cudaError_t topk_grid(K kern, int threads, int smem, int64_t rows, int* grid_out) {
    const int sms = current_sms();
    cudaError_t e = set_smem_attr((const void*)kern, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > rows) grid = rows;
    *grid_out = (int)grid;
    return cudaSuccess;
}

cudaError_t topk_rows_launch(const float* logits, int64_t rows, int S, int Skv, int ratio,
                             const int32_t* ks, const int32_t* ke, int topk, int32_t* out_idx,
                             float* out_sc, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    int grid = 0;
    const int smem = (int)sizeof(TopkSmemRows);
    cudaError_t e = topk_grid(topk_rows_kernel, kTopkRowThreads, smem, rows, &grid);
    if (e != cudaSuccess) return e;
    topk_rows_kernel<<<(unsigned)grid, kTopkRowThreads, smem, stream>>>(logits, rows, S, Skv, ratio, ks,
                                                                        ke, topk, out_idx, out_sc);
    return cudaGetLastError();
}

cudaError_t topk_rows_bf16_launch(const uint16_t* scores, int64_t rows, int S, int Skv, const int2* urange,
                                  int QT, int topk, int32_t* out_idx, uint16_t* out_sc, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    int grid = 0;
    const int smem = (int)sizeof(TopkSmemBf16);
    cudaError_t e = topk_grid(topk_rows_bf16_kernel, kTopkBf16Threads, smem, rows, &grid);
    if (e != cudaSuccess) return e;
    topk_rows_bf16_kernel<<<(unsigned)grid, kTopkBf16Threads, smem, stream>>>(scores, rows, S, Skv, urange, QT,
                                                                              topk, out_idx, out_sc);
    return cudaGetLastError();
}

LIDX_STATUS_READER(status_misc)

}  // namespace lidx
