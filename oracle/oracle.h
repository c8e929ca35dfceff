/*
 * oracle.h -- plain, slow CPU reference of the lightning-indexer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * links it, includes it or calls it, and the two share no code.
 *
 * Arithmetic is fp64 over bf16-decoded inputs unless a function says
 * otherwise.  Rows are indexed r = b*S + s.  Layouts follow the indexer pages:
 *   V4   ("tilelang_indexer", V4IndexerFunction docstring):
 *        q [S,B,H,D] bf16, k [Skv,B,D] bf16, w [S,B,H] fp32
 *   V4.1 ("deepseek_v41.indexer", indexer_scores parameters):
 *        q [B,S,H,D] bf16, k [B,Skv,D] bf16, w [B,S,H] bf16, allowed [B,S,Skv] u8
 * bf16 tensors are passed as their raw 16-bit patterns.
 */
#ifndef LIDX_ORACLE_H
#define LIDX_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_ACT_RELU = 0, ORC_ACT_IDENTITY = 1 };

void orc_set_threads(int n);
int orc_get_threads(void);

/* bf16 pattern -> double, and double -> nearest-even bf16 value. */
double orc_bf16_decode(uint16_t v);
double orc_bf16_round(double v);
void orc_bf16_round_array(const double* in, double* out, int64_t n);

/* _make_causal_cu_seqlens: ks[s] = 0, ke[s] = min((s+1)//ratio, Skv). */
void orc_causal_ranges(int64_t S, int64_t Skv, int ratio, int32_t* ks, int32_t* ke);

/* batched_indexer_fwd / indexer_fwd_interface for a list of rows:
 * out[i, t] = sum_h w[s,b,h] * act(q[s,b,h,:] . k[t,b,:]) for ks[s] <= t < ke[s],
 * -inf elsewhere.  out is [nrows, Skv]. */
int orc_logits_rows(const uint16_t* q, const uint16_t* k, const float* w,
                    int64_t B, int64_t S, int64_t Skv, int H, int D,
                    const int32_t* ks, const int32_t* ke, int act,
                    const int64_t* rows, int64_t nrows, double* out);

/* Per-row top-k over the visible range [ks[s], ke[s]) of each logits row:
 * sorted by score descending, equal scores by ascending index; when fewer
 * than topk keys are visible the tail is index -1 / score -inf. */
int orc_topk_rows(const double* logits, int64_t nrows, int64_t Skv,
                  const int64_t* rows, int64_t S, const int32_t* ks, const int32_t* ke,
                  int topk, int32_t* idx_out, double* score_out);

/* Per-row top-k over the entries whose mask byte is nonzero (the V4.1
 * selection over visible keys): same order and padding as orc_topk_rows.
 * logits and mask are [nrows, Skv]. */
int orc_topk_masked_rows(const double* logits, const uint8_t* mask, int64_t nrows, int64_t Skv,
                         int topk, int32_t* idx_out, double* score_out);

/* pytorch_extract_topk_scores: out[i,j] = logits[i, idx[i,j]], -inf for an
 * index outside [0, Skv). */
void orc_extract_rows(const double* logits, int64_t nrows, int64_t Skv,
                      const int32_t* idx, int topk, double* out);

/* Scores of given (row, index) pairs without a dense sweep:
 * out[i,j] = sum_h w*act(q.k[idx]) when ks[s] <= idx < ke[s], else -inf. */
int orc_gather_scores_rows(const uint16_t* q, const uint16_t* k, const float* w,
                           int64_t B, int64_t S, int64_t Skv, int H, int D,
                           const int32_t* ks, const int32_t* ke, int act,
                           const int64_t* rows, int64_t nrows,
                           const int32_t* idx /*[nrows,topk]*/, int topk, double* out);

/* V4.1 indexer_scores for a list of rows (r = b*S + s):
 * y = bf16(q.k), z = bf16(act(y) * w), out = bf16(sum_h z) where allowed,
 * -inf elsewhere.  The bf16 result is returned as a float.  out [nrows, Skv]. */
int orc_scores_v41_rows(const uint16_t* q, const uint16_t* k, const uint16_t* w,
                        const uint8_t* allowed, int64_t B, int64_t S, int64_t Skv,
                        int H, int D, int act, const int64_t* rows, int64_t nrows,
                        float* out);

/* V4IndexerFunction.backward through the selected entries.  For each row and
 * slot j with ks <= t = idx < ke and g = grad[j]:
 *   dw[s,b,h] += g*act(x);  c = g*w*act'(x);  dq[s,b,h,:] += c*k[t];  dk[t,b,:] += c*q[s,b,h,:]
 * with x = q[s,b,h,:].k[t,b,:].  All outputs are overwritten.  The *_slack
 * outputs (nullable) accumulate |contribution| of pairs whose ReLU decision is
 * within float32 accumulation error (|x| <= gamma * sum_d |q_d k_d|). */
int orc_bwd(const uint16_t* q, const uint16_t* k, const float* w,
            const int32_t* idx, const float* grad,
            int64_t B, int64_t S, int64_t Skv, int H, int D,
            const int32_t* ks, const int32_t* ke, int topk, int act, double gamma,
            double* dq, double* dk, double* dw,
            double* dq_slack, double* dk_slack, double* dw_slack);

#ifdef __cplusplus
}
#endif
#endif
