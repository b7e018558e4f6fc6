/*
 * headloss_lmhead.h -- the LM-head GEMM in front of the loss (C ABI).
 *
 * The monolithic head loss consumes the logits of the language-model head,
 * logits = hidden . weight^T (ServiceNow Fast-LLM PR #549, "Correctness":
 * the LM head and tied embeddings are among the axes the head loss is
 * validated on).  This call computes that GEMM on the GB300's 5th-generation
 * tensor cores and, in the same pass, the per-row softmax statistics of each
 * 256-column tile of its output -- the statistics a loss's first pass would
 * otherwise read the logits back to compute.  It is the first building block
 * of a fused LM head; the loss calls of headloss.h do not use it yet.
 *
 * Status codes are those of headloss.h.
 */
#ifndef HEADLOSS_LMHEAD_H
#define HEADLOSS_LMHEAD_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * headloss_lmhead_logits -- logits and per-tile row statistics.
 *
 * hidden:  N x D bf16, row-major, device, 16-byte aligned base.
 * weight:  V x D bf16, row-major, device, 16-byte aligned base (one row per
 *          vocabulary entry).
 * N, D, V: N a multiple of 128, V a multiple of 256, D a multiple of 64.
 * logits:  N x V bf16, row-major, device, 16-byte aligned (written):
 *          the fp32 sum over D of hidden[i, :] * weight[j, :], rounded once
 *          to bf16 (round to nearest even).
 * stats:   N x (V / 256) pairs of fp32, device, 8-byte aligned (written): for row i and
 *          column tile k, (m, s) with m = max over the tile's 256 bf16
 *          logits and s = sum of exp(logit - m) over them.  The row's
 *          log-sum-exp is m* + log(sum_k s_k * exp(m_k - m*)), m* = max_k m_k.
 * err:     one int in device memory (4-byte aligned), zeroed by the caller:
 *          bit 0 is set if a wait inside the kernel gave up (a copy or an MMA
 *          did not complete within ~2 s); the kernel then stops issuing work,
 *          waits for what it issued, and the outputs are unreliable.
 * stream:  cudaStream_t (NULL = legacy default stream).  Asynchronous.
 *
 * The kernel is persistent (one CTA per SM over the 128 x 256 output
 * tiles): tcgen05.mma on bf16 operands staged by TMA, fp32 accumulation in
 * two TMEM accumulators (one tile's epilogue overlaps the next tile's MMAs),
 * logits written by TMA stores from shared memory.
 *
 * Returns HEADLOSS_OK, HEADLOSS_ERR_ARG (a size not a multiple above, or a
 * null pointer), HEADLOSS_ERR_ALIGN (a base not 16-byte aligned, stats not
 * 8-byte or err not 4-byte aligned) or
 * HEADLOSS_ERR_CUDA (tensor-map encoding or launch failed).  The caller owns
 * every buffer; the call allocates nothing.
 */
int headloss_lmhead_logits(const void* hidden, const void* weight, int N, int D, int V,
                           void* logits, void* stats, int* err, void* stream);

/*
 * headloss_lmhead_logits_rowstats -- the same GEMM with, per (row, 256-column
 * tile), the loss's first-pass record of the tile instead of (m, s): the
 * statistics headloss_forward_backward_rowstats (include/headloss.h) consumes.
 *
 * softcap, logits_scale: those of the loss handle that will consume the
 *            statistics (softcap c >= 0, 0 = off; logits_scale s > 0).  For a
 *            teacher's logits: softcap 0 and logits_scale 1 / T (the teacher
 *            enters the loss as t / T).
 * temperature: the distillation temperature T > 0 of the consuming handle;
 *            read only when row_stats_t is non-null.
 * row_stats: N x (V / 256) records of 4 fp32, device, 16-byte aligned
 *            (written): for the bf16 logits x of row i and tile k, with
 *            zs = s c tanh(x / c) log2(e) (c = 0: zs = s x log2(e)),
 *            (m2, S, E, X): m2 = max zs, S = sum 2^(zs - m2),
 *            E = sum 2^(zs - m2) (zs - m2), X = max |x| (exact: the largest
 *            magnitude among the tile's bf16 logits).
 * row_stats_t: null, or N x (V / 256) fp32 (device, 4-byte aligned,
 *            written): S_T = sum 2^((zs - m2) / T) per tile, which a student
 *            row needs for the distillation losses when T != 1 (one more
 *            exponential per logit in the epilogue).
 * Other arguments, checks and errors as headloss_lmhead_logits (ERR_ARG also
 * for a negative or non-finite softcap, a non-positive logits_scale, or a
 * non-positive or non-finite temperature with row_stats_t; ERR_ALIGN for a
 * misaligned row_stats_t).
 */
int headloss_lmhead_logits_rowstats(const void* hidden, const void* weight, int N, int D, int V,
                                    float softcap, float logits_scale, float temperature,
                                    void* logits, void* row_stats, float* row_stats_t, int* err,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HEADLOSS_LMHEAD_H */
