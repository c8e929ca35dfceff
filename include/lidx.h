/*
 * lidx.h -- C ABI of the GB300 (sm_103a) lightning-indexer library, liblidx.so.
 *
 * The lightning indexer scores every (query s, compressed key t) pair with
 *     score[b,s,t] = sum_h w[.,h] * act(q[s,b,h,:] . k[t,b,:])
 * masks it causally on compressed positions (or with an explicit visibility
 * tensor), and keeps the top-k keys per query row.  Sources (indexer
 * documentation pages):
 *   [P1] "nemo_automodel...deepseek_v4.kernels.tilelang_indexer":
 *        V4IndexerFunction (layouts q [S,B,H,D] bf16, k [Skv,B,D] bf16,
 *        weights [S,B,H] fp32; forward(index_q, index_k, weights,
 *        compress_ratio, topk, topk_indices=None); backward(grad_scores,
 *        grad_indices)), v4_lighting_indexer (returns [B,S,topk] fp32),
 *        pytorch_extract_topk_scores(logits, topk_indices).
 *   [P2] "nemo_automodel...deepseek_v4.kernels.tilelang_indexer_fwd":
 *        _make_causal_cu_seqlens (query p sees groups [0,(p+1)//compress_ratio)),
 *        batched_indexer_fwd / indexer_fwd_interface ([S,Skv] fp32 logits over
 *        cu_seqlen_ks..cu_seqlen_ke, clean_logits=True), clean_logits_.
 *   [P3] "nemo_automodel...deepseek_v41.indexer": indexer_scores(queries
 *        [B,S,H,D] bf16, keys [B,Skv,D] bf16, weights [B,S,H] bf16, allowed
 *        [B,S,Skv] bool) -> bf16 [B,S,Skv]; GEMM result and weighted head score
 *        rounded to bf16 before an fp32 head reduction.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers on the current CUDA device unless the
 *     argument says "host".  The caller owns every buffer; the library never
 *     allocates device memory (its only device state is a file-scope status
 *     word).  Inputs are read-only; outputs are fully overwritten (padding
 *     included) unless stated.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronising.  A nonzero return means
 *     nothing was launched, except LIDX_ERR_CUDA (a launch failed).
 *   - Argument rules (checked before any launch, LIDX_ERR_SHAPE otherwise):
 *     H a power of two <= 128 and D a multiple of 16 [P3 queries parameter],
 *     here also D <= 128; B, S >= 1; Skv >= 0; compress_ratio >= 1; topk >= 1
 *     where a top-k is asked for.  Base pointers of bf16/fp32 tensors must be
 *     16-byte aligned (LIDX_ERR_ALIGN); tensors are dense and contiguous in the
 *     stated layout.  NULL where a buffer is required -> LIDX_ERR_NULL.
 *   - Inputs must be finite; NaN or inf inputs give unspecified (but
 *     in-bounds) results.
 *   - Device-side failures (a pipeline wait that exceeds its time limit) are
 *     recorded in the status word read by lidx_device_status().
 */
#ifndef LIDX_H
#define LIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LIDX_OK = 0,
    LIDX_ERR_NULL = 1,        /* required pointer is NULL */
    LIDX_ERR_SHAPE = 2,       /* size/shape rule violated */
    LIDX_ERR_ALIGN = 3,       /* pointer not 16-byte aligned */
    LIDX_ERR_UNSUPPORTED = 4, /* valid request outside what this build implements */
    LIDX_ERR_WORKSPACE = 5,   /* workspace too small (see lidx_workspace_bytes) */
    LIDX_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
    LIDX_ERR_DEVICE_TIMEOUT = 7, /* a kernel gave up on a pipeline wait */
    LIDX_ERR_NO_DEVICE = 8    /* no sm_103a device current */
} lidx_status;

typedef enum { LIDX_ACT_RELU = 0, LIDX_ACT_IDENTITY = 1 } lidx_act;

/* Operation ids for lidx_workspace_bytes. */
typedef enum {
    LIDX_OP_INDEXER_FWD = 0,
    LIDX_OP_INDEXER_BWD = 1,
    LIDX_OP_SCORES_V41 = 2,
    LIDX_OP_TOPK_V41 = 3
} lidx_op;

/*
 * V4 forward: causal mask + per-row top-k   [P1 V4IndexerFunction.forward,
 * v4_lighting_indexer; P2 _make_causal_cu_seqlens].
 *   q  bf16 [S,B,H,D]   k bf16 [Skv,B,D]   w fp32 [S,B,H]   (SBHD, row-major)
 *   Row (b,s) sees keys t in [0, min((s+1)/compress_ratio, Skv)).
 *   logits_out  fp32 [B,S,Skv], nullable.  Non-NULL: every entry is written,
 *               masked ones as -inf, and the top-k reads it back.  NULL: the
 *               logits are never written to HBM (fused path; needs workspace).
 *   topk_indices_in  int32 [B,S,topk], nullable.  Non-NULL: no selection; the
 *               scores of the given indices are returned (entries outside the
 *               row's visible range give -inf) and indices_out is a copy.  The
 *               scores come from the same tensor-core sweep of the row's
 *               visible keys (needs the workspace unless logits_out is given).
 *   indices_out int32 [B,S,topk]  scores_out fp32 [B,S,topk]: sorted by score
 *               descending, equal scores by ascending index; rows with fewer
 *               than topk visible keys end with index -1 / score -inf.
 *   workspace   device scratch of lidx_workspace_bytes(LIDX_OP_INDEXER_FWD,..)
 *               bytes (may be NULL when that is 0), 256-byte aligned.
 *   Limit of this build: Skv <= 65536 when a selection is made (no limit with
 *   topk_indices_in).
 */
int lidx_indexer_fwd(const void* q, const void* k, const float* w,
                     int64_t B, int64_t S, int64_t Skv, int H, int D,
                     int compress_ratio, int topk, int act,
                     const int32_t* topk_indices_in, float* logits_out,
                     int32_t* indices_out, float* scores_out,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * V4 forward over explicit per-row ranges   [P2 batched_indexer_fwd /
 * indexer_fwd_interface: cu_seqlen_ks, cu_seqlen_ke; P1 forward].  As
 * lidx_indexer_fwd, except that row (b,s) sees keys t in
 * [max(ks[s],0), min(ke[s],Skv)) instead of the causal range.  ks, ke: int32
 * [S] device arrays, both required.  A context-parallel rank holding query
 * rows [p0, p0+S) of a longer sequence, with every compressed key gathered
 * [P3 indexer_scores, keys], passes ks = 0 and ke = min((p0+s+1)/compress_ratio,
 * Skv) and gets exactly the rows of the unsharded call.
 */
int lidx_indexer_fwd_ranges(const void* q, const void* k, const float* w,
                            int64_t B, int64_t S, int64_t Skv, int H, int D,
                            const int32_t* ks, const int32_t* ke, int topk, int act,
                            const int32_t* topk_indices_in, float* logits_out,
                            int32_t* indices_out, float* scores_out,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The fused forward of lidx_indexer_fwd (logits not written, selection made)
 * without a caller-supplied workspace.  The indexer pages have no counterpart:
 * this call exists for callers that cannot allocate device memory (code that
 * runs inside an allocator or memory-pool callback, in a process whose device
 * memory is reserved up front by another framework, or in a plug-in that only
 * receives input and output pointers).  Its scratch is one array inside the
 * library of lidx_noalloc_scratch_bytes() bytes (24 MiB), held on every GPU
 * that loads the library until the process exits.  Arguments and outputs are
 * those of lidx_indexer_fwd.  Returns LIDX_ERR_WORKSPACE when the call would
 * need more scratch than the array holds (lidx_workspace_bytes(...) >
 * lidx_noalloc_scratch_bytes(); e.g. at H=64 about 2*4*Skv*4 bytes per SM).
 * The first call on a device looks up the array's address; make it before any
 * stream capture.  Calls share the array: calls that overlap on the GPU race.
 */
int lidx_indexer_fwd_noalloc(const void* q, const void* k, const float* w,
                             int64_t B, int64_t S, int64_t Skv, int H, int D,
                             int compress_ratio, int topk, int act,
                             int32_t* indices_out, float* scores_out, void* stream);

/* Size in bytes of the scratch array lidx_indexer_fwd_noalloc uses. */
size_t lidx_noalloc_scratch_bytes(void);

/*
 * Logits only, explicit ranges   [P2 batched_indexer_fwd, indexer_fwd_interface,
 * clean_logits_].  Same layouts as lidx_indexer_fwd.
 *   ks, ke  int32 [S] (device), nullable together: NULL -> causal ranges from
 *           compress_ratio.  Row (b,s) sees t in [max(ks[s],0), min(ke[s],Skv)).
 *   clean   1: entries outside the range are -inf.  0: entries outside the
 *           range are unspecified (left as they were or holding raw scores).
 *   logits_out fp32 [B,S,Skv].
 */
int lidx_indexer_logits(const void* q, const void* k, const float* w,
                        int64_t B, int64_t S, int64_t Skv, int H, int D,
                        int compress_ratio, const int32_t* ks, const int32_t* ke,
                        int clean, int act, float* logits_out, void* stream);

/*
 * Gather at indices   [P1 pytorch_extract_topk_scores(logits, topk_indices)].
 *   logits fp32 [B,S,Skv]; idx int32 [B,S,topk]; scores_out fp32 [B,S,topk] =
 *   logits[b,s,idx], -inf where idx is outside [0,Skv).  Bit-exact copy.
 */
int lidx_extract_topk_scores(const float* logits, const int32_t* idx,
                             int64_t B, int64_t S, int64_t Skv, int topk,
                             float* scores_out, void* stream);

/*
 * Per-row top-k of given logits   [P1 forward with topk_indices=None: the
 * selection step; P2 cu_seqlen_ks/cu_seqlen_ke ranges].
 *   logits fp32 [rows, Skv] row-major, rows = B*S; row r is query s = r % S.
 *   ks, ke int32 [S] (device), nullable together: NULL -> causal ranges
 *   [0, min((s+1)/compress_ratio, Skv)).  Only entries in the row's range are
 *   candidates.  Output as lidx_indexer_fwd: indices_out int32 / scores_out
 *   fp32 [rows, topk], sorted by score descending, ties by ascending index,
 *   padded with -1 / -inf.  Limit of this build: Skv <= 65536.
 */
int lidx_topk_rows(const float* logits, int64_t rows, int64_t S, int64_t Skv,
                   int compress_ratio, const int32_t* ks, const int32_t* ke, int topk,
                   int32_t* indices_out, float* scores_out, void* stream);

/*
 * V4.1 scores   [P3 indexer_scores, module docstring].
 *   q bf16 [B,S,H,D]  k bf16 [B,Skv,D]  w bf16 [B,S,H]  allowed u8/bool [B,S,Skv]
 *   scores_out bf16 [B,S,Skv]: where allowed[b,s,t] != 0,
 *       bf16( sum_h  bf16( act(bf16(q.k)) * w ) )   (fp32 head reduction),
 *   and -inf (0xFF80) elsewhere.  allowed needs no alignment.
 *   workspace: lidx_workspace_bytes(LIDX_OP_SCORES_V41, ...) bytes, 256-byte aligned.
 */
int lidx_indexer_scores_v41(const void* q, const void* k, const void* w,
                            const uint8_t* allowed, int64_t B, int64_t S, int64_t Skv,
                            int H, int D, int act, void* scores_out,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * V4.1 scores and their per-row top-k   [P3 indexer_scores; module docstring:
 * the top-k / candidate selection runs on these scores].  Scores as
 * lidx_indexer_scores_v41; then, per row (b,s), the top `topk` of the visible
 * keys (allowed != 0) by bf16 score, sorted descending, equal scores by
 * ascending key index; rows with fewer visible keys end with index -1 /
 * score -inf.
 *   scores_out      bf16 [B,S,Skv], nullable: NULL keeps the scores in the
 *                   workspace instead.
 *   indices_out     int32 [B,S,topk];  topk_scores_out bf16 [B,S,topk].
 *   workspace       lidx_workspace_bytes(LIDX_OP_TOPK_V41, B,S,Skv,H,D,topk,
 *                   scores_out != NULL) bytes, 256-byte aligned.
 *   Visible scores must be finite (they are for finite inputs of this size).
 *   Limit of this build: Skv <= 65536.
 */
int lidx_indexer_topk_v41(const void* q, const void* k, const void* w,
                          const uint8_t* allowed, int64_t B, int64_t S, int64_t Skv,
                          int H, int D, int act, int topk, void* scores_out,
                          int32_t* indices_out, void* topk_scores_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * V4 backward through the selected entries   [P1 V4IndexerFunction.backward;
 * grad_indices carries no gradient and is not an argument].
 *   idx int32 [B,S,topk] (as returned by the forward), grad_scores fp32
 *   [B,S,topk].  Slots with idx outside the row's causal range (padding -1
 *   included) contribute nothing.  For every other slot, with t = idx,
 *   g = grad, x = q[s,b,h,:].k[t,b,:]:
 *     dw[s,b,h] += g*act(x);  dq[s,b,h,:] += g*w*act'(x)*k[t,b,:];
 *     dk[t,b,:] += sum_h g*w*act'(x)*q[s,b,h,:]        (ReLU'(0) = 0)
 *   dq [S,B,H,D] and dk [Skv,B,D]: fp32 when grad_dtype = 0, bf16 (each the
 *   fp32 result rounded to nearest even) when grad_dtype = 1; dw fp32 [S,B,H].
 *   All are overwritten.  No atomic operation touches them: two calls on the
 *   same inputs give identical bits.  Limit of this build: Skv <= 65536.
 *   workspace: lidx_workspace_bytes(LIDX_OP_INDEXER_BWD, ...) bytes.
 */
int lidx_indexer_bwd(const void* q, const void* k, const float* w,
                     const int32_t* idx, const float* grad_scores,
                     int64_t B, int64_t S, int64_t Skv, int H, int D,
                     int compress_ratio, int topk, int act, int grad_dtype,
                     void* dq, void* dk, float* dw,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward over explicit per-row ranges (the ranges of lidx_indexer_fwd_ranges):
 * as lidx_indexer_bwd, with slot t of row (b,s) contributing only when
 * max(ks[s],0) <= t < min(ke[s],Skv).  A context-parallel rank gets its own
 * rows' dq and dw and a partial dk; the ranks' partial dk sum to the full dk.
 */
int lidx_indexer_bwd_ranges(const void* q, const void* k, const float* w,
                            const int32_t* idx, const float* grad_scores,
                            int64_t B, int64_t S, int64_t Skv, int H, int D,
                            const int32_t* ks, const int32_t* ke, int topk, int act,
                            int grad_dtype, void* dq, void* dk, float* dw,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Device scratch the call needs for these sizes, in bytes (0 = none).
 * logits_materialised: 1 if logits_out will be non-NULL (LIDX_OP_INDEXER_FWD). */
size_t lidx_workspace_bytes(int op, int64_t B, int64_t S, int64_t Skv, int H, int D,
                            int topk, int logits_materialised);

/* Synchronises `stream`, returns the device status word (LIDX_OK or
 * LIDX_ERR_DEVICE_TIMEOUT) and clears it.  LIDX_ERR_CUDA if the sync fails. */
int lidx_device_status(void* stream);

/*
 * Failure-detection controls (no counterpart on the pages).  Every pipeline
 * wait inside the kernels gives up after a time limit, records
 * LIDX_ERR_DEVICE_TIMEOUT in the status word and winds its kernel down, so a
 * stalled pipeline ends the launch instead of hanging the GPU.
 *   lidx_set_wait_limit_ns  sets that limit for later launches (0 restores the
 *                           default of 2 s) and returns the previous one.
 *   lidx_debug_stall_producer  1: later launches of the scoring kernels (V4,
 *                           V4.1) and of the backward's tensor-core kernels
 *                           load nothing, so their waits run out (for tests of
 *                           the timeout path; outputs are then unspecified);
 *                           0: normal operation.  Returns the previous setting.
 * Both are process-wide and take effect at the next launch.
 */
uint64_t lidx_set_wait_limit_ns(uint64_t ns);
int lidx_debug_stall_producer(int on);

/* Static English description of a status code (never NULL). */
const char* lidx_status_string(int status);

/* Library version, e.g. 0x000200 for 0.2.0. */
int lidx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LIDX_H */
