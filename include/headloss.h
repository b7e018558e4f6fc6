/*
 * headloss.h -- C ABI of the fused language-model head loss (GB300, sm_103a).
 *
 * One call reads each token row of vocabulary logits, computes its softmax
 * statistics once, and shares them across every requested loss and metric:
 * label cross-entropy, z-loss, distillation (from-distribution CE, forward KL,
 * reverse KL, with temperature), the GRPO clipped objective with its
 * ratio / KL / clamp / advantage statistics, and entropy.  In the same pass it
 * writes one combined logits gradient and every requested scalar.
 *
 * Source of the operation (ServiceNow Fast-LLM pages):
 *   - issue #507 "Monolithic fused head-loss kernel", Problem / Proposed
 *     direction: a flag set of losses and metrics, one softmax, all scalars
 *     and the combined gradient in one pass;
 *   - PR #549 "Monolithic fused head-loss kernel (torch.compile)", Approach
 *     and Loss coverage: the loss set, one logits scale per softmax, fp32
 *     gradient accumulation cast to the logits dtype once;
 *   - PR #558 "Triton monolithic kernel", Design: the gradient is a per-row
 *     superposition  grad_j = prob_coeff * softmax_j - label_coeff * delta(j, label),
 *     extended here by a teacher term and a reverse-KL log-ratio term;
 *     Validation: masking, logit / gradient scaling, softcap, metrics without
 *     gradient.
 *
 * Conventions shared by every entry point:
 *   - Every call returns an int status (HEADLOSS_OK == 0).  On any error no
 *     device work has been enqueued and no output was touched.
 *   - The caller owns every buffer.  All data pointers are DEVICE pointers of
 *     the current CUDA device.
 *   - headloss_forward_backward is asynchronous on `stream`: it never
 *     synchronises the host and never allocates.  Results are valid after the
 *     stream is synchronised.
 *   - One handle may be used by one stream at a time (it owns a small
 *     workspace for per-cluster partial sums).
 */
#ifndef HEADLOSS_H
#define HEADLOSS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same layout as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* headloss_stream_t;

typedef struct headloss* headloss_t;

/* Logits dtype: the teacher logits and the gradient have the same dtype. */
enum headloss_dtype { HEADLOSS_FP32 = 0, HEADLOSS_BF16 = 1, HEADLOSS_FP16 = 2 };

/* Loss / metric selection.  A flag selects EMISSION of the scalar; the
 * matching weight selects its GRADIENT contribution (weight 0 = metric only,
 * PR #558 "metrics-without-gradient"). */
enum headloss_flag {
    HEADLOSS_CE = 1u << 0,          /* label cross-entropy, lse - z[label] */
    HEADLOSS_Z = 1u << 1,           /* z-loss, lse^2 */
    HEADLOSS_DIST_CE = 1u << 2,     /* -sum_j q_j log pT_j (teacher q, student pT at T) */
    HEADLOSS_FKL = 1u << 3,         /* KL(q || pT) */
    HEADLOSS_RKL = 1u << 4,         /* KL(pT || q) */
    HEADLOSS_GRPO = 1u << 5,        /* -min(rho A, clip(rho, 1-eps, 1+eps) A) */
    HEADLOSS_GRPO_STATS = 1u << 6,  /* new_logprob / ratio / clip / KL / advantage stats */
    HEADLOSS_ENTROPY = 1u << 7      /* H(p) of the student softmax */
};

enum headloss_status {
    HEADLOSS_OK = 0,
    HEADLOSS_ERR_ARG = 1,           /* bad size, flag, weight, temperature, ... */
    HEADLOSS_ERR_DTYPE = 2,         /* dtype not one of enum headloss_dtype */
    HEADLOSS_ERR_ALIGN = 3,         /* a logits / teacher / gradient base not 16-byte aligned */
    HEADLOSS_ERR_MISSING_INPUT = 4, /* a flag's required input pointer is NULL */
    HEADLOSS_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    HEADLOSS_ERR_TIMEOUT = 6,       /* device: a bounded wait for a row copy gave up */
    HEADLOSS_ERR_LABEL_RANGE = 7,   /* device: a label >= V (that row was treated as masked) */
    HEADLOSS_ERR_SIZE = 8           /* V too large for the on-chip row plan of this dtype/flag set */
};

/* Loss weights.  grad_scale multiplies the whole gradient (the incoming
 * gradient of the total loss); it does not scale the emitted scalars. */
typedef struct {
    float ce, z, dist_ce, fkl, rkl, grpo, entropy, grad_scale;
} headloss_weights;

/* Scalar slots of scalars_out (16 floats).  Means are over valid rows.
 * Slots of losses / metrics not selected by the flags are written 0. */
enum headloss_slot {
    HEADLOSS_SLOT_TOTAL = 0,        /* sum over selected losses of weight * mean */
    HEADLOSS_SLOT_CE = 1,
    HEADLOSS_SLOT_Z = 2,
    HEADLOSS_SLOT_DIST_CE = 3,
    HEADLOSS_SLOT_FKL = 4,
    HEADLOSS_SLOT_RKL = 5,
    HEADLOSS_SLOT_GRPO = 6,
    HEADLOSS_SLOT_NEW_LOGPROB = 7,  /* mean of z[label] - lse */
    HEADLOSS_SLOT_RATIO = 8,        /* mean of rho = exp(new - old log-prob) */
    HEADLOSS_SLOT_CLIP_FRAC = 9,    /* fraction of rows with |rho - 1| > eps */
    HEADLOSS_SLOT_KL_K3 = 10,       /* mean of rho - 1 - log rho */
    HEADLOSS_SLOT_ADV_MEAN = 11,
    HEADLOSS_SLOT_ADV_STD = 12,     /* population standard deviation */
    HEADLOSS_SLOT_ENTROPY = 13,
    HEADLOSS_SLOT_N_VALID = 14,     /* exact integer (exact while < 2^24) */
    HEADLOSS_SLOT_N_CLIPPED = 15    /* exact integer (exact while < 2^24) */
};

/*
 * headloss_create -- validate a loss set and build a handle.
 *
 * flags:        OR of enum headloss_flag (at least one bit; unknown bits -> ERR_ARG).
 * w:            weights (NULL = all loss weights 0 except ce = grpo = 1, grad_scale = 1).
 *               A weight of a loss whose flag is not set is ignored.
 * temperature:  T > 0, divides student AND teacher logits for the three
 *               distillation losses only (PR #549 "Bundled fix": the
 *               distillation temperature is honoured).  At T = 2 exactly,
 *               streamed bf16 teacher rows without softcap or entropy take
 *               the probabilities at T = 1 and at T from one exponential
 *               (2^d = (2^(d/2))^2): the same results within the stated
 *               tolerances, fewer operations per element.
 * clip_eps:     GRPO epsilon >= 0 (symmetric clip).
 * softcap:      c >= 0; c > 0 applies z = c * tanh(x / c) before the scale.
 * logits_scale: s > 0; the student softmax sees z = s * softcap(x) (PR #549
 *               Approach: one softmax, one logits_scale_factor).
 * out:          receives the handle.
 *
 * Allocates the handle's workspace on the current device (the only
 * allocation this library makes).  Errors: ERR_ARG, ERR_CUDA.
 */
int headloss_create(uint32_t flags, const headloss_weights* w, float temperature,
                    float clip_eps, float softcap, float logits_scale, headloss_t* out);

/*
 * headloss_forward_backward -- one fused pass over N rows of V logits.
 *
 * logits:         N x V, row-major, contiguous, `dtype`; base 16-byte aligned
 *                 (rows need not be: a row whose bytes are not a multiple of 16
 *                 is handled with element-wise edges).
 * labels:         N int64 (NULL = no labels: every row valid; CE / GRPO /
 *                 GRPO_STATS then return ERR_MISSING_INPUT).  label < 0 masks
 *                 the row for every loss and metric: its gradient row is
 *                 written as exact +0 and it is not counted.  label >= V is a
 *                 device error (ERR_LABEL_RANGE via headloss_get_device_error)
 *                 and that row is treated as masked.
 * teacher_logits: N x V, same layout and dtype (required by DIST_CE / FKL /
 *                 RKL, else ignored).
 * old_logprobs:   N fp32 old-policy log-probs of the label (GRPO, GRPO_STATS).
 * advantages:     N fp32 per-token advantages (GRPO, GRPO_STATS).
 * grad_out:       N x V, `dtype`, 16-byte aligned, or NULL for metrics only.
 *                 It may equal `logits` (in-place; such a call always uses
 *                 the resident kernel, whatever plan is pinned, and returns
 *                 ERR_SIZE where a row does not fit on chip); it must not
 *                 overlap the teacher.  Written: d(grad_scale * total) / d logits, where
 *                 total = sum_k weight_k * mean_over_valid_rows(loss_k).
 * scalars_out:    16 fp32 (enum headloss_slot).
 * stream:         CUDA stream for all device work.
 *
 * N == 0 is valid (no input is read; every scalar is written 0).
 *
 * Errors (host-side, nothing enqueued): ERR_ARG (N < 0, V < 1, V >= 2^31,
 * null handle / scalars_out, null logits with N > 0), ERR_DTYPE, ERR_ALIGN,
 * ERR_MISSING_INPUT (N > 0 only), ERR_SIZE, ERR_CUDA (launch failure).
 */
int headloss_forward_backward(headloss_t h, const void* logits, int64_t N, int64_t V, int dtype,
                              const int64_t* labels, const void* teacher_logits,
                              const float* old_logprobs, const float* advantages,
                              void* grad_out, float* scalars_out, headloss_stream_t stream);

/*
 * Optional per-call extras of headloss_forward_backward_ext.  Zero-initialise
 * the struct and set only what is needed; an all-zero struct (or a NULL
 * pointer) gives exactly headloss_forward_backward.
 *
 * new_logprobs:  N fp32 (device) or NULL.  log p(label) of the student
 *                softmax at T = 1 for every row: the GRPO "new_logprobs"
 *                output of the fused head loss (Fast-LLM PR #549, "Loss
 *                coverage").  Masked rows get 0.  Requires labels.
 * row_loss:      N fp32 (device) or NULL.  The row's total loss,
 *                sum_k weight_k * loss_k(row) over the selected losses, whose
 *                mean over valid rows is scalars_out[HEADLOSS_SLOT_TOTAL] (per
 *                token losses for callers that weight tokens themselves).
 *                Masked rows get 0.
 * accumulate:    0 writes grad_out; 1 adds this call's gradient to the values
 *                already in grad_out (the sum formed in the kernel's compute
 *                precision -- fp32 for 16-bit logits, fp64 for fp32 logits --
 *                then one rounding to the output dtype), as in gradient accumulation
 *                across micro-batches (PR #558, "Validation").  Masked rows
 *                keep their values.  grad_out must not overlap the logits.
 * divisor:       > 0: the normaliser of a batch split over several calls
 *                (PR #549, "Correctness": cross-entropy splits).  It replaces
 *                the call's own valid-row count in the gradient scale and in
 *                the loss slots (TOTAL, CE, Z, DIST_CE, FKL, RKL, GRPO,
 *                ENTROPY), so that the gradients and loss slots of the calls
 *                that make up a batch add up to those of the whole batch when
 *                every call passes the batch's valid-row count.  The metric
 *                slots (NEW_LOGPROB .. ADV_STD, N_VALID, N_CLIPPED) stay over
 *                the call's own rows.  0: the call's own count.  Must be
 *                finite.
 * token_coeff:   N fp32 (device) or NULL.  A per-row coefficient c_i =
 *                d(total)/d(log p(label_i)) computed outside the call -- GSPO's
 *                per-token coefficient from headloss_gspo_seam -- superposed on
 *                the gradient as c_i (delta(j, label) - p_j) on the label
 *                column the label-based losses share (PR #558, "Design": the
 *                GSPO seam hands the kernel a per-token coefficient that
 *                superposes with the in-kernel losses).  grad_scale does not
 *                multiply it (the seam already did).  Masked rows ignore it.
 *                Requires labels; such a call uses the resident kernel.
 */
typedef struct {
    float* new_logprobs;
    float* row_loss;
    int accumulate;
    double divisor;
    const float* token_coeff;
} headloss_call_ext;

/*
 * headloss_forward_backward_ext -- headloss_forward_backward with the extras
 * above (the arguments before `ext` are those of headloss_forward_backward).
 * Extra errors (host-side, nothing enqueued): ERR_ARG (divisor < 0 or not
 * finite, accumulate with grad_out NULL or overlapping the logits), ERR_ALIGN
 * (new_logprobs / row_loss / token_coeff not 4-byte aligned),
 * ERR_MISSING_INPUT (new_logprobs or token_coeff without labels, N > 0).
 */
int headloss_forward_backward_ext(headloss_t h, const void* logits, int64_t N, int64_t V,
                                  int dtype, const int64_t* labels, const void* teacher_logits,
                                  const float* old_logprobs, const float* advantages,
                                  void* grad_out, float* scalars_out,
                                  const headloss_call_ext* ext, headloss_stream_t stream);

/*
 * headloss_get_device_error -- synchronise `stream`, then read and clear the
 * handle's device error word.  *err receives HEADLOSS_OK, ERR_LABEL_RANGE or
 * ERR_TIMEOUT (the first of those raised since the last read).
 */
int headloss_get_device_error(headloss_t h, headloss_stream_t stream, int* err);

/* The two row kernels a plan may use. */
enum headloss_kernel {
    HEADLOSS_KERNEL_AUTO = 0,
    /* A thread-block cluster holds each row in shared memory (each CTA a
     * column slice, statistics merged over DSMEM): every byte of logits is
     * read from HBM once.  Any dtype, any V up to its shared-memory limit. */
    HEADLOSS_KERNEL_RESIDENT = 1,
    /* One CTA streams each row through a ring of chunk slots twice
     * (statistics, then gradient in reverse chunk order so the second read
     * finds the row in L2).  bf16 / fp16 rows whose bytes are a multiple of 16. */
    HEADLOSS_KERNEL_STREAM = 2
};

/* A launch plan.  In headloss_force_plan a zero field leaves that choice to
 * the planner. */
typedef struct {
    int kernel;      /* enum headloss_kernel */
    int cluster;     /* resident: CTAs per row, 1..8 (streaming: 1) */
    int stages;      /* resident: row stages per CTA, 1..4; streaming: chunk slots, 2..8 */
    int threads;     /* threads per CTA: 256 or 512 */
    int chunk_words; /* streaming: 16-byte words per thread per chunk: 1, 2 or 4 */
} headloss_plan_desc;

/*
 * headloss_plan -- the plan a call with (V, dtype) would use, the CTAs it
 * launches and its dynamic shared memory per CTA.  Any output may be NULL.
 * Errors: ERR_ARG, ERR_DTYPE, ERR_SIZE, ERR_CUDA.
 */
int headloss_plan(headloss_t h, int64_t V, int dtype, headloss_plan_desc* plan, int* ctas,
                  int* smem_bytes);

/*
 * headloss_force_plan -- pin some or all plan choices for later calls on this
 * handle (NULL: back to the automatic plan).  For tests and tuning.  A call
 * whose rows cannot use the pinned choices returns ERR_SIZE.  Errors: ERR_ARG.
 */
int headloss_force_plan(headloss_t h, const headloss_plan_desc* plan);

/*
 * headloss_forward_backward_noalloc -- headloss_forward_backward without a
 * handle and without any device allocation, for callers that cannot allocate
 * when they compute the loss: inside a CUDA-graph capture (allocation is not
 * allowed there), under a memory pool that forbids raw cudaMalloc, or in a
 * loop that must never touch the allocator.  (The pages describe no such
 * entry point; it is an addition of this library.)
 *
 * Arguments: the configuration of headloss_create followed by the arguments
 * of headloss_forward_backward, with the same meanings, layouts and checks.
 *
 * Scratch: instead of a handle's workspace it uses one fixed device array in
 * the library (1024 partial-sum slots + a count and an error word, 131,328
 * bytes), present on every device that loads the library until the process
 * exits.  Launches are planned to use at most those 1024 slots; a launch that
 * would need more returns HEADLOSS_ERR_SIZE.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address once; make that first call before any stream
 * capture.  Every call shares the array and overwrites what it uses (the
 * count and partial sums are rewritten by each call, the error word is
 * cleared on `stream` first), so calls on different streams that overlap on
 * the GPU race with one another: order them on one stream.  Device-side
 * conditions (a label >= V, a copy timeout) are not reported to the caller by
 * this entry point; such rows are treated as masked.  Never calls cudaMalloc,
 * cudaFree or any allocating routine.
 */
int headloss_forward_backward_noalloc(uint32_t flags, const headloss_weights* w, float temperature,
                                      float clip_eps, float softcap, float logits_scale,
                                      const void* logits, int64_t N, int64_t V, int dtype,
                                      const int64_t* labels, const void* teacher_logits,
                                      const float* old_logprobs, const float* advantages,
                                      void* grad_out, float* scalars_out, headloss_stream_t stream);

/*
 * headloss_gspo_seam -- GSPO's per-segment seam: the sequence-level ratio,
 * its clipped objective and the per-token coefficient the backward call
 * superposes (headloss_call_ext.token_coeff).  GSPO runs in three steps, as
 * in ServiceNow Fast-LLM PR #558 "Design" (forward, eager segment seam,
 * load-mode backward) and PR #549 "Loss coverage":
 *   1. headloss_forward_backward_ext with new_logprobs (grad_out may be NULL);
 *   2. this call;
 *   3. headloss_forward_backward_ext with token_coeff (and the other losses).
 * The objective: segment i is rows [seg_offsets[i], seg_offsets[i+1]); over
 * its valid rows T_i (0 <= label < V; L_i of them)
 *   s_i = exp((1/L_i) sum_t (new_t - old_t))   (geometric mean of token ratios)
 *   A_i = mean of advantages_t over T_i
 *   obj_i = min(s_i A_i, clip(s_i, 1 - clip_eps, 1 + clip_eps) A_i)
 * and the loss is -(1/G) sum_i obj_i over the G segments that hold a valid
 * row.  The unclipped branch carries the gradient unless it is the larger
 * objective (ties count as unclipped).
 *
 * new_logprobs:  N fp32 (device): log p(label) per row at T = 1 (step 1).
 * old_logprobs:  N fp32, advantages: N fp32 (one advantage per sequence
 *                broadcast to its rows), labels: N int64 -- all device.
 * N, V:          rows and vocabulary size (V decides which labels are valid).
 * seg_offsets:   n_seg + 1 int64 (device), non-decreasing from 0 to N.
 *                Offsets outside [0, N] are clamped and a decreasing pair is
 *                an empty segment; overlapping segments are not detected.
 * clip_eps:      >= 0.  weight, grad_scale: finite; the coefficient is that
 *                of weight * grad_scale * loss.
 * token_coeff:   N fp32 (device, written): c_t = d(weight * grad_scale *
 *                loss)/d(new_t) = -weight * grad_scale * A_i s_i / (G L_i)
 *                for a valid row of a segment on its unclipped branch, else 0.
 * scalars_out:   4 fp32 (device, written): loss, mean s_i, fraction of
 *                segments with |s_i - 1| > clip_eps, G.
 * Two launches on `stream`, deterministic (fp64, fixed-order sums); no
 * allocation.  Errors (nothing enqueued): ERR_ARG (N < 0, V < 1, n_seg < 1,
 * clip_eps < 0, a non-finite weight, a NULL pointer), ERR_ALIGN (fp32 arrays
 * not 4-byte, int64 arrays not 8-byte aligned), ERR_CUDA.
 */
int headloss_gspo_seam(const float* new_logprobs, const float* old_logprobs,
                       const float* advantages, const int64_t* labels, int64_t N, int64_t V,
                       const int64_t* seg_offsets, int n_seg, float clip_eps, float weight,
                       float grad_scale, float* token_coeff, float* scalars_out,
                       headloss_stream_t stream);

/*
 * headloss_forward_backward_rowstats -- the loss of headloss_forward_backward
 * from logits whose first-pass statistics the LM-head GEMM already produced
 * (headloss_lmhead_logits_rowstats in include/headloss_lmhead.h): one read of
 * the logits (and the teacher's) and one write of the gradient per row, no
 * statistics pass.  The fused LM head of ServiceNow Fast-LLM PR #549
 * ("Correctness": the LM head and tied embeddings) computes the head GEMM and
 * the loss back to back; on GB300 the GEMM's epilogue emits each output
 * tile's share of the softmax statistics from TMEM.
 *
 * Arguments as headloss_forward_backward, plus:
 * row_stats:     N x (V / 256) records of 4 fp32 (device, 16-byte aligned)
 *                from headloss_lmhead_logits_rowstats called with this
 *                handle's softcap and logits_scale on the same logits.
 * row_stats_t:   with a teacher and temperature T != 1: the same call's
 *                N x (V / 256) sums at T (row_stats_t there, 4-byte aligned);
 *                null otherwise (at T = 1 the records' S serve).
 * teacher_stats: with a teacher: N x (V / 256) records from
 *                headloss_lmhead_logits_rowstats on the teacher's logits with
 *                softcap 0 and logits_scale 1 / T (16-byte aligned); null
 *                otherwise.
 * Losses: CE, Z, GRPO, GRPO_STATS, ENTROPY, and with a teacher DIST_CE and
 * FKL (their values are summed during the pass: the gradient needs no cross
 * sum).  REVERSE KL is refused (ERR_ARG): its coefficient needs the cross sum
 * of pT (log pT - log q) before the pass.  dtype must be HEADLOSS_BF16
 * (ERR_DTYPE) and V a multiple of 256 (ERR_ARG); a missing teacher_stats, or
 * row_stats_t at T != 1, is ERR_MISSING_INPUT.  In place is allowed (each
 * word is read before its gradient replaces it).  Three launches; results as
 * headloss_forward_backward, within the same tolerances.
 * ext:           NULL, or the extras of headloss_forward_backward_ext with
 *                the same meaning and errors: per-row log p(label) and total
 *                loss, accumulation into grad_out (not in place), the
 *                divisor of a split batch, and GSPO's per-token coefficient.
 *                With ext, GSPO runs on the GEMM's records as well: this call
 *                with new_logprobs (grad_out may be NULL), headloss_gspo_seam,
 *                then this call with token_coeff.
 */
int headloss_forward_backward_rowstats(headloss_t h, const void* logits, int64_t N, int64_t V,
                                       int dtype, const int64_t* labels,
                                       const void* teacher_logits, const float* old_logprobs,
                                       const float* advantages, const void* row_stats,
                                       const float* row_stats_t, const void* teacher_stats,
                                       void* grad_out, float* scalars_out,
                                       const headloss_call_ext* ext, headloss_stream_t stream);

/* Kernel launches one headloss_forward_backward call enqueues (constant). */
int headloss_launches_per_call(void);

void headloss_destroy(headloss_t h);
const char* headloss_strerror(int status);
int headloss_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HEADLOSS_H */
