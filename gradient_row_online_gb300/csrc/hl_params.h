// hl_params.h -- launch parameters shared by the host planner and the kernels.
#pragma once
#include <stdint.h>

namespace hl {

// Compile-time feature set of one row-kernel instantiation.
enum : int {
    F_TEACH = 1,    // teacher row + student-at-temperature sums (DIST_CE / FKL / RKL)
    F_RKL = 2,      // reverse-KL sum and its log-ratio gradient term
    F_ENT = 4,      // entropy sum (metric and/or gradient)
    F_SOFTCAP = 8,  // z = s * c * tanh(x / c)
    // streaming kernel only (the resident kernels take FEAT & F_BASE):
    F_DCE = 16,     // teacher-entropy sum for the from-distribution CE
    F_ENTG = 32,    // entropy gradient term (entropy weight nonzero)
    F_BASE = 15,
    // host-side only: the call adds its gradient to grad_out (selects the
    // accumulating instantiation, which carries F_DCE / F_ENTG whenever
    // F_TEACH / F_ENT)
    F_ACC = 64,
    // fp32 row kernel only: per-element arithmetic in double-float (fp32
    // pairs) instead of fp64; for student-only rows without softcap whose
    // gradient has no entropy term (the entropy may still be a metric)
    F_DF = 128,
    // streaming kernel only: L2 cache hints on the row copies (the teacher's
    // first pass evict-last, second pass evict-first); for teacher rows
    // without softcap, where it measured faster (the second read then hits L2
    // more often).  Every teacher instantiation stores its gradient with the
    // streaming hint.
    F_L2P = 256,
    // streaming kernel only: the distillation temperature is exactly 2, so
    // a logit's probabilities at T = 1 and at T share one exponential:
    // 2^d = (2^(d/2))^2 (bf16 teacher rows without softcap or entropy)
    F_T2 = 512,
};

// Loss / metric bits (values match enum headloss_flag).
enum : uint32_t {
    L_CE = 1u, L_Z = 2u, L_DIST_CE = 4u, L_FKL = 8u, L_RKL = 16u,
    L_GRPO = 32u, L_GRPO_STATS = 64u, L_ENTROPY = 128u,
};

// Device error bits (read back by headloss_get_device_error).
enum : int { E_LABEL = 1, E_TIMEOUT = 2 };

constexpr int THREADS = 512;  // maximum threads per CTA (a plan may launch 256)
constexpr int NWARPS = THREADS / 32;
constexpr int MAX_CLUSTER = 8;
constexpr int MAX_STAGES = 8;          // mbarrier slots (streaming ring)
constexpr int MAX_RESIDENT_STAGES = 4; // row stages of the resident kernel

// Partial-statistics record one CTA contributes for one row (all base-2
// units; see the row kernel for definitions).
enum Rec { R_ZM, R_UM, R_S, R_E, R_ST, R_SQ, R_EQ, R_XP, R_Y, R_ZY, R_HASY, NREC };

// Per-cluster partial sums over its rows (fp64), reduced by the finalize kernel.
enum Acc {
    A_CE, A_Z, A_DCE, A_FKL, A_RKL, A_GRPO, A_LP, A_RATIO, A_KL3, A_ADV, A_ADV2,
    A_ENT, A_NVALID, A_NCLIP, NACC_USED
};
constexpr int NACC = 16;

struct Params {
    const void* x;         // N x V logits
    const void* t;         // N x V teacher logits (or null)
    void* g;               // N x V gradient (or null)
    const int64_t* labels; // N (or null)
    const float* old_lp;   // N (or null)
    const float* adv;      // N (or null)
    int64_t N, V;
    int64_t L;             // columns per CTA slice (multiple of 16 bytes' worth)
    int C;                 // CTAs per cluster (one row per cluster)
    int nbuf;              // row stages buffered per CTA
    int words;             // 16-byte words per operand stage buffer
    uint32_t flags;
    float s, softcap, T, eps;
    float w_ce, w_z, w_dce, w_fkl, w_rkl, w_grpo, w_ent, grad_scale;
    double* partials;              // [clusters][NACC]
    const long long* n_valid;      // valid-row count of this call
    const float* kscale;           // grad_scale / (divisor or valid-row count), set by the count kernel
    int* err;                      // device error word
    unsigned long long wait_ns;    // limit of every mbarrier wait (~2 s)
    int64_t drop_row;              // fault-injection builds only: row whose copy is skipped (-1: none)
    float* lp_out;                 // N per-row log p(label) (or null)
    float* rl_out;                 // N per-row total loss (or null)
    double divisor;                // > 0: normaliser replacing the valid-row count
    int accumulate;                // 1: add the gradient to grad_out's values
    const float* tok;              // N per-row d(total)/d(log p(label)) added on the label
                                   // column (GSPO's per-token coefficient), or null
};

}  // namespace hl
