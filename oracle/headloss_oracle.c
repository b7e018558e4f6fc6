/*
 * headloss_oracle.c -- plain fp64 CPU oracle for the monolithic LM-head loss.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (ServiceNow Fast-LLM pages):
 *   - issue #507 "Monolithic fused head-loss kernel", Problem and Proposed
 *     direction: one softmax per token row shared by label cross-entropy,
 *     z-loss, distillation, the GRPO clipped objective with its
 *     ratio / KL / clamp / advantage statistics, and entropy; every scalar
 *     plus the combined logits gradient.
 *   - PR #549, Loss coverage: from-distribution CE, forward KL and reverse KL
 *     with temperature; GRPO objective + new_logprobs + metric family +
 *     entropy.  Bundled fix: distillation honours its temperature.
 *   - PR #549, Approach: one logits scale per softmax (logits_scale_factor).
 *   - PR #549 Correctness / PR #558 Validation: masking, logit and gradient
 *     scaling, softcap, metrics without gradient.
 *
 * The pages print no loss formula.  Every loss below is the textbook
 * definition the pages' names imply, under these readings: softcap
 * z = s * c * tanh(x / c) (c = 0: off), gradient with respect to raw x;
 * label < 0 masks a row for every loss; temperature divides student and
 * teacher for the distillation losses only, no T^2 factor; means over the
 * valid rows of the call; GRPO ratio at T = 1 with a symmetric clip, the
 * unclipped branch carrying the gradient unless it is the larger objective
 * (ties count as unclipped); clip fraction |rho - 1| > eps, k3 = rho - 1 -
 * log rho; entropy H(p) of the student at T = 1.  The gradient is written out term by term
 * from each loss's own definition -- NOT from the per-row coefficient
 * superposition of PR #558 "Design" -- so that superposition is what the
 * tests check the CUDA path against.
 *
 * Everything is fp64, one row at a time, in the most direct form.  Rows are
 * independent, so an OpenMP loop over rows is the only parallelism.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* loss / metric selection bits (same meaning as the library's flags, but
 * defined independently here) */
#define OR_CE 1u
#define OR_Z 2u
#define OR_DIST_CE 4u
#define OR_FKL 8u
#define OR_RKL 16u
#define OR_GRPO 32u
#define OR_GRPO_STATS 64u
#define OR_ENTROPY 128u
#define OR_DIST_ANY (OR_DIST_CE | OR_FKL | OR_RKL)

typedef struct {
    uint32_t flags;
    double w_ce, w_z, w_dist_ce, w_fkl, w_rkl, w_grpo, w_entropy;
    double grad_scale;
    double temperature; /* distillation temperature T > 0 */
    double clip_eps;    /* GRPO clip epsilon >= 0 */
    double softcap;     /* c; 0 disables */
    double logits_scale;/* s > 0 */
} oracle_cfg;

/* Per-row record written by oracle_rows (all zero for a masked row). */
enum {
    RF_VALID = 0,  /* 1 for a row that counts, 0 for a masked row */
    RF_CE,         /* lse - z_label */
    RF_Z,          /* lse^2 */
    RF_DIST_CE,    /* -sum q log pT */
    RF_FKL,        /* sum q (log q - log pT) */
    RF_RKL,        /* sum pT (log pT - log q) */
    RF_GRPO,       /* -min(rho A, clip(rho) A) */
    RF_LOGPROB,    /* new log-prob of the label, z_y - lse */
    RF_RATIO,      /* rho = exp(logprob - old_logprob) */
    RF_CLIPPED,    /* 1 when |rho - 1| > eps */
    RF_KL3,        /* rho - 1 - log rho */
    RF_ADV,        /* A */
    RF_ADV2,       /* A^2 */
    RF_ENTROPY,    /* -sum p log p */
    RF_AMBIGUOUS,  /* 1 when log rho lies within 1e-5 of log(1 +- eps) */
    RF_ACT,        /* 1 when the unclipped GRPO branch carries the gradient */
    RF_LSE,        /* lse, for diagnostics */
    RF_COUNT
};

#define ORACLE_AMBIGUITY 1e-5

int oracle_row_fields(void) { return RF_COUNT; }

/* Softcap then scale, the head-output reading: z = s * c * tanh(x / c). */
static double transform(const oracle_cfg* cfg, double x) {
    double y = cfg->softcap > 0.0 ? cfg->softcap * tanh(x / cfg->softcap) : x;
    return cfg->logits_scale * y;
}

/* dz/dx of the transform above: s * (1 - tanh^2(x / c)), evaluated as
 * s / cosh^2(x / c) -- the same quantity without the cancellation of
 * 1 - tanh^2 where tanh saturates (cosh overflow gives the exact limit 0). */
static double transform_deriv(const oracle_cfg* cfg, double x) {
    if (cfg->softcap > 0.0) {
        const double ch = cosh(x / cfg->softcap);
        return cfg->logits_scale / (ch * ch);
    }
    return cfg->logits_scale;
}

/* log sum_j exp(a_j), written with the usual max shift. */
static double log_sum_exp(const double* a, int64_t n) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (a[j] > m) m = a[j];
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s += exp(a[j] - m);
    return m + log(s);
}

int64_t oracle_count_valid(const int64_t* labels, int64_t n_rows) {
    if (!labels) return n_rows;
    int64_t n = 0;
    for (int64_t i = 0; i < n_rows; ++i)
        if (labels[i] >= 0) ++n;
    return n;
}

/*
 * One row.  x, t: V logits (fp64, exact upcasts of the inputs); label < 0
 * masks the row.  inv_n = 1 / (valid rows of the whole call).
 * rec: RF_COUNT fields.  grad (nullable): dL/dx for this row, where
 * L = grad_scale * sum_k w_k * mean_over_valid_rows(loss_k).
 * gmag (nullable): the size of the quantities dL/dx is computed from (sum over
 * loss terms of |term|, where a factor that is itself a difference counts its
 * parts): the scale at which rounding error of a superposed gradient lives.
 */
static void oracle_row(const oracle_cfg* cfg, int64_t V, const double* x, int64_t label,
                       int has_labels, const double* t, double old_lp, double adv,
                       double inv_n, double* rec, double* grad, double* gmag,
                       double* work /* 6 * V */) {
    const uint32_t f = cfg->flags;
    memset(rec, 0, sizeof(double) * RF_COUNT);
    int valid = !has_labels || label >= 0;
    if (!valid) {
        if (grad) memset(grad, 0, sizeof(double) * V);
        if (gmag) memset(gmag, 0, sizeof(double) * V);
        return;
    }
    rec[RF_VALID] = 1.0;

    double* z = work;          /* transformed student logits */
    double* p = work + V;      /* softmax(z) */
    double* zT = work + 2 * V; /* z / T */
    double* pT = work + 3 * V; /* softmax(z / T) */
    double* u = work + 4 * V;  /* t / T */
    double* q = work + 5 * V;  /* softmax(t / T) */

    for (int64_t j = 0; j < V; ++j) z[j] = transform(cfg, x[j]);
    const double lse = log_sum_exp(z, V);
    for (int64_t j = 0; j < V; ++j) p[j] = exp(z[j] - lse);
    rec[RF_LSE] = lse;

    double lse_T = 0.0, lsq = 0.0;
    const int dist = (f & OR_DIST_ANY) != 0;
    if (dist) {
        const double T = cfg->temperature;
        for (int64_t j = 0; j < V; ++j) zT[j] = z[j] / T;
        lse_T = log_sum_exp(zT, V);
        for (int64_t j = 0; j < V; ++j) pT[j] = exp(zT[j] - lse_T);
        for (int64_t j = 0; j < V; ++j) u[j] = t[j] / T;
        lsq = log_sum_exp(u, V);
        for (int64_t j = 0; j < V; ++j) q[j] = exp(u[j] - lsq);
    }

    /* ---- forward: each loss from its definition ---- */
    double zy = 0.0;
    if (has_labels) zy = z[label];
    if (f & OR_CE) rec[RF_CE] = lse - zy;
    if (f & OR_Z) rec[RF_Z] = lse * lse;
    double rkl = 0.0;
    if (dist) {
        double dce = 0.0, fkl = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            const double log_pT = zT[j] - lse_T;
            const double log_q = u[j] - lsq;
            dce -= q[j] * log_pT;
            fkl += q[j] * (log_q - log_pT);
            rkl += pT[j] * (log_pT - log_q);
        }
        if (f & OR_DIST_CE) rec[RF_DIST_CE] = dce;
        if (f & OR_FKL) rec[RF_FKL] = fkl;
        if (f & OR_RKL) rec[RF_RKL] = rkl;
    }
    double H = 0.0;
    if (f & OR_ENTROPY) {
        for (int64_t j = 0; j < V; ++j)
            if (p[j] > 0.0) H -= p[j] * (z[j] - lse);
        rec[RF_ENTROPY] = H;
    }
    /* GRPO: policy ratio of the label token against the old policy. */
    double rho = 0.0, act = 0.0;
    if (f & (OR_GRPO | OR_GRPO_STATS)) {
        const double eps = cfg->clip_eps;
        const double lp = zy - lse;
        rho = exp(lp - old_lp);
        double rho_c = rho;
        if (rho_c < 1.0 - eps) rho_c = 1.0 - eps;
        if (rho_c > 1.0 + eps) rho_c = 1.0 + eps;
        const double unclipped = rho * adv, clipped = rho_c * adv;
        /* loss = -min(unclipped, clipped) */
        const double obj = unclipped < clipped ? unclipped : clipped;
        /* Which branch carries d(loss)/d(rho): the unclipped one unless the
         * clipped value is strictly smaller, and the clamp passes the
         * gradient at its end points (torch.clamp / torch.minimum ties). */
        if (unclipped <= clipped) act = 1.0;
        else act = (rho >= 1.0 - eps && rho <= 1.0 + eps) ? 1.0 : 0.0;
        rec[RF_GRPO] = -obj;
        rec[RF_LOGPROB] = lp;
        rec[RF_RATIO] = rho;
        rec[RF_CLIPPED] = fabs(rho - 1.0) > eps ? 1.0 : 0.0;
        rec[RF_KL3] = rho - 1.0 - (lp - old_lp);
        rec[RF_ADV] = adv;
        rec[RF_ADV2] = adv * adv;
        rec[RF_ACT] = act;
        const double lr = lp - old_lp;
        int amb = fabs(lr - log(1.0 + eps)) < ORACLE_AMBIGUITY;
        if (1.0 - eps > 0.0 && fabs(lr - log(1.0 - eps)) < ORACLE_AMBIGUITY) amb = 1;
        rec[RF_AMBIGUOUS] = amb ? 1.0 : 0.0;
    }

    if (!grad && !gmag) return;

    /* ---- backward: d/dz_j of each weighted mean loss, one term per loss ---- */
    const double k = cfg->grad_scale * inv_n;
    const double T = cfg->temperature;
    for (int64_t j = 0; j < V; ++j) {
        const double delta = (has_labels && j == label) ? 1.0 : 0.0;
        /* terms[i]: one loss's contribution; mags[i]: the size of the
         * quantities it is computed from (a factor that is itself a
         * difference, like log pT - log q - RKL, counts its parts, down to
         * the logits and row log-sum-exps a log-probability is formed from:
         * log pT_j = zT_j - lse_T) */
        double terms[8], mags[8];
        int nt = 0;
        /* CE: d(lse - z_y)/dz_j = p_j - delta */
        if (f & OR_CE) {
            terms[nt] = k * cfg->w_ce * (p[j] - delta);
            mags[nt++] = fabs(k * cfg->w_ce) * (p[j] + delta);
        }
        /* z-loss: d(lse^2)/dz_j = 2 lse p_j */
        if (f & OR_Z) {
            terms[nt] = k * cfg->w_z * 2.0 * lse * p[j];
            mags[nt] = fabs(terms[nt]);
            ++nt;
        }
        /* from-distribution CE: d(-sum_i q_i log pT_i)/dz_j = (pT_j - q_j) / T */
        if (f & OR_DIST_CE) {
            terms[nt] = k * cfg->w_dist_ce * (pT[j] - q[j]) / T;
            mags[nt++] = fabs(k * cfg->w_dist_ce / T) * (pT[j] + q[j]);
        }
        /* forward KL: sum q log q does not depend on z, same derivative */
        if (f & OR_FKL) {
            terms[nt] = k * cfg->w_fkl * (pT[j] - q[j]) / T;
            mags[nt++] = fabs(k * cfg->w_fkl / T) * (pT[j] + q[j]);
        }
        /* reverse KL: d/dz_j sum_i pT_i (log pT_i - log q_i)
         *           = pT_j (log pT_j - log q_j - RKL) / T */
        if (f & OR_RKL) {
            const double log_pT = zT[j] - lse_T, log_q = u[j] - lsq;
            terms[nt] = k * cfg->w_rkl * pT[j] * (log_pT - log_q - rkl) / T;
            mags[nt++] = fabs(k * cfg->w_rkl * pT[j] / T) *
                         (fabs(zT[j]) + fabs(lse_T) + fabs(u[j]) + fabs(lsq) + fabs(rkl));
        }
        /* GRPO: d loss/d rho = -A (unclipped branch) or 0; d rho/d lp = rho;
         * d lp/dz_j = delta - p_j */
        if (f & OR_GRPO) {
            terms[nt] = k * cfg->w_grpo * (-adv * act) * rho * (delta - p[j]);
            mags[nt++] = fabs(k * cfg->w_grpo * adv * act * rho) * (delta + p[j]);
        }
        /* entropy: dH/dz_j = -p_j (log p_j + H) */
        if (f & OR_ENTROPY) {
            terms[nt] = k * cfg->w_entropy * (-p[j] * ((z[j] - lse) + H));
            mags[nt++] = fabs(k * cfg->w_entropy * p[j]) * (fabs(z[j]) + fabs(lse) + fabs(H));
        }

        const double dzdx = transform_deriv(cfg, x[j]);
        double g = 0.0, mag = 0.0;
        for (int i = 0; i < nt; ++i) {
            g += terms[i];
            mag += mags[i];
        }
        if (grad) grad[j] = g * dzdx;
        if (gmag) gmag[j] = mag * fabs(dzdx);
    }
}

/*
 * Rows [0, n_rows) of a call whose valid-row count is n_valid_total.
 * x, t: n_rows x V row-major fp64 (t may be NULL when no distillation flag is
 * set); labels may be NULL (every row valid).  old_lp / adv: n_rows entries or
 * NULL.  rec: n_rows x RF_COUNT.  grad / gmag: n_rows x V or NULL.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_rows(const oracle_cfg* cfg, int64_t n_rows, int64_t V, const double* x,
                const int64_t* labels, const double* t, const double* old_lp,
                const double* adv, int64_t n_valid_total, double* rec, double* grad,
                double* gmag, int n_threads) {
    if (n_rows < 0 || V <= 0 || !x || !rec) return -1;
    const uint32_t f = cfg->flags;
    if ((f & OR_DIST_ANY) && !t) return -1;
    if ((f & (OR_CE | OR_GRPO | OR_GRPO_STATS)) && !labels) return -1;
    if ((f & (OR_GRPO | OR_GRPO_STATS)) && (!old_lp || !adv)) return -1;
    if (labels)
        for (int64_t i = 0; i < n_rows; ++i)
            if (labels[i] >= V) return -1;
    const double inv_n = n_valid_total > 0 ? 1.0 / (double)n_valid_total : 0.0;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double* work = (double*)malloc(sizeof(double) * 6 * (size_t)V);
        if (!work) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (int64_t i = 0; i < n_rows; ++i) {
                oracle_row(cfg, V, x + i * V, labels ? labels[i] : 0, labels != NULL,
                           t ? t + i * V : NULL, old_lp ? old_lp[i] : 0.0,
                           adv ? adv[i] : 0.0, inv_n, rec + i * RF_COUNT,
                           grad ? grad + i * V : NULL, gmag ? gmag + i * V : NULL, work);
            }
            free(work);
        }
    }
    (void)n_threads;
    return bad ? -1 : 0;
}

/* Neumaier-compensated sum of a[i * stride + field] over n_rows. */
static double column_sum(const double* rec, int64_t n_rows, int field) {
    double s = 0.0, c = 0.0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const double v = rec[i * RF_COUNT + field];
        const double tsum = s + v;
        if (fabs(s) >= fabs(v)) c += (s - tsum) + v;
        else c += (v - tsum) + s;
        s = tsum;
    }
    return s + c;
}

/*
 * The sixteen scalars of a call from its per-row records (fp64):
 *  0 total = sum over flagged losses of weight * mean loss
 *  1 ce  2 z  3 dist_ce  4 fkl  5 rkl  6 grpo_loss
 *  7 new_logprob_mean  8 ratio_mean  9 clip_frac  10 kl_k3  11 adv_mean
 *  12 adv_std (population)  13 entropy_mean  14 n_valid  15 n_clipped
 * Means are over valid rows; with no valid row every mean is 0.  Slots of
 * losses / metrics that are not flagged are 0.
 */
void oracle_reduce(const oracle_cfg* cfg, const double* rec, int64_t n_rows, double* out16) {
    const uint32_t f = cfg->flags;
    for (int i = 0; i < 16; ++i) out16[i] = 0.0;
    const double n = column_sum(rec, n_rows, RF_VALID);
    out16[14] = n;
    if (n <= 0.0) return;
#define MEAN(field) (column_sum(rec, n_rows, (field)) / n)
    if (f & OR_CE) out16[1] = MEAN(RF_CE);
    if (f & OR_Z) out16[2] = MEAN(RF_Z);
    if (f & OR_DIST_CE) out16[3] = MEAN(RF_DIST_CE);
    if (f & OR_FKL) out16[4] = MEAN(RF_FKL);
    if (f & OR_RKL) out16[5] = MEAN(RF_RKL);
    if (f & OR_GRPO) out16[6] = MEAN(RF_GRPO);
    if (f & OR_GRPO_STATS) {
        out16[7] = MEAN(RF_LOGPROB);
        out16[8] = MEAN(RF_RATIO);
        out16[9] = MEAN(RF_CLIPPED);
        out16[10] = MEAN(RF_KL3);
        const double am = MEAN(RF_ADV);
        const double var = MEAN(RF_ADV2) - am * am;
        out16[11] = am;
        out16[12] = var > 0.0 ? sqrt(var) : 0.0;
        out16[15] = column_sum(rec, n_rows, RF_CLIPPED);
    }
    if (f & OR_ENTROPY) out16[13] = MEAN(RF_ENTROPY);
#undef MEAN
    double total = 0.0;
    if (f & OR_CE) total += cfg->w_ce * out16[1];
    if (f & OR_Z) total += cfg->w_z * out16[2];
    if (f & OR_DIST_CE) total += cfg->w_dist_ce * out16[3];
    if (f & OR_FKL) total += cfg->w_fkl * out16[4];
    if (f & OR_RKL) total += cfg->w_rkl * out16[5];
    if (f & OR_GRPO) total += cfg->w_grpo * out16[6];
    if (f & OR_ENTROPY) total += cfg->w_entropy * out16[13];
    out16[0] = total;
}

/* A whole call: per-row records, gradient and the sixteen scalars. */
int oracle_forward_backward(const oracle_cfg* cfg, int64_t n_rows, int64_t V, const double* x,
                            const int64_t* labels, const double* t, const double* old_lp,
                            const double* adv, double* grad, double* gmag, double* rec,
                            double* out16, int n_threads) {
    const int64_t n_valid = oracle_count_valid(labels, n_rows);
    int rc = oracle_rows(cfg, n_rows, V, x, labels, t, old_lp, adv, n_valid, rec, grad, gmag,
                         n_threads);
    if (rc) return rc;
    oracle_reduce(cfg, rec, n_rows, out16);
    return 0;
}
