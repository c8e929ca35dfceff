// noalloc.cu -- the fused V4 forward for callers that cannot allocate device
// memory.
//
// The fused forward (score + causal mask + top-k without writing logits)
// needs a scratch area for its per-CTA row buffers.  lidx_indexer_fwd takes
// that area from the caller.  Some callers have no way to provide it: code
// that runs where cudaMalloc is not allowed or not wanted (inside a custom
// allocator or memory-pool callback, in a process whose device memory is
// fully reserved up front by another framework, or in a plug-in that is
// handed only input and output pointers).  This entry point serves them with
// a scratch array that lives in the library itself.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Its
// device address is looked up once per device with cudaGetSymbolAddress (the
// host-side name of the array is only a stand-in, never a device pointer);
// that lookup happens on the first call on each device, so make the first
// call before any stream capture.  All calls share the one array: calls that
// overlap on the GPU (different streams, or different host threads) race on it
// and must be serialised by the caller.  The kernel writes every scratch entry
// it later reads, so nothing has to be cleared between calls.  The looked-up
// address is kept for the life of the process: a caller that resets a device
// (cudaDeviceReset) must not call this entry point on that device again.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "lidx.h"

namespace lidx {

constexpr size_t kNoAllocScratchBytes = (size_t)24 << 20;  // 24 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once).
static int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LIDX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LIDX_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return LIDX_OK;
}

}  // namespace lidx

extern "C" size_t lidx_noalloc_scratch_bytes(void) { return lidx::kNoAllocScratchBytes; }

extern "C" int lidx_indexer_fwd_noalloc(const void* q, const void* k, const float* w, int64_t B,
                                        int64_t S, int64_t Skv, int H, int D, int compress_ratio,
                                        int topk, int act, int32_t* indices_out, float* scores_out,
                                        void* stream) {
    // the same rules as lidx_indexer_fwd apply, checked first; only the scratch source differs
    const int rc0 = lidx::check_fwd(q, k, w, B, S, Skv, H, D, compress_ratio, nullptr, nullptr, topk,
                                    act, nullptr, nullptr, indices_out, scores_out);
    if (rc0 != LIDX_OK) return rc0;
    const size_t need = lidx_workspace_bytes(LIDX_OP_INDEXER_FWD, B, S, Skv, H, D, topk, 0);
    if (need > lidx::kNoAllocScratchBytes) return LIDX_ERR_WORKSPACE;  // beyond the static array
    void* scratch = nullptr;
    if (need > 0) {
        const int rc = lidx::noalloc_scratch(&scratch);
        if (rc != LIDX_OK) return rc;
    }
    return lidx_indexer_fwd(q, k, w, B, S, Skv, H, D, compress_ratio, topk, act, nullptr, nullptr,
                            indices_out, scores_out, scratch, need > 0 ? lidx::kNoAllocScratchBytes : 0,
                            stream);
}
