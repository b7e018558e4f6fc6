// headloss_api.cu -- the C ABI (include/headloss.h): argument checks, the
// launch planner, and the two small kernels around the row kernel (valid-row
// count before it, deterministic scalar finalize after it).
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "headloss.h"
#include "hl_params.h"
#include "hl_rows.cuh"

namespace hl {
const void* rows_kernel_bf16(int feat);
const void* rows_kernel_fp16(int feat);
const void* rows_kernel_fp32(int feat);
const void* stream_kernel_bf16(int feat);
const void* stream_kernel_fp16(int feat);
const void* rows_kernel_bf16_acc(int feat);
const void* rows_kernel_fp16_acc(int feat);
const void* stream_kernel_bf16_acc(int feat);
const void* stream_kernel_fp16_acc(int feat);
const void* onepass_kernel_bf16(int feat);
int onepass_smem_bytes();

// Valid rows of the call (0 <= label < V); a label >= V raises E_LABEL.
// One block: the count is an exact integer whatever the order.
// It also stores the gradient factor grad_scale / (divisor, else the count)
// once for the row kernels, as an fp32 quotient (fp64 division is slow here
// and this kernel runs ahead of the row kernel).
__global__ void __launch_bounds__(1024) count_valid_kernel(const int64_t* labels, int64_t N,
                                                           int64_t V, long long* out, int* err,
                                                           float grad_scale, double divisor,
                                                           float* kscale) {
    __shared__ long long part[32];
    // the row kernel may start now; it waits for this grid before it reads
    // the count
    asm volatile("griddepcontrol.launch_dependents;");
    long long c = 0;
    int bad = 0;
    if (labels) {
        for (int64_t i = threadIdx.x; i < N; i += blockDim.x) {
            const int64_t y = labels[i];
            if (y >= 0 && y < V) ++c;
            else if (y >= V) bad = 1;
        }
    } else if (threadIdx.x == 0) {
        c = N;
    }
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    if (bad) atomicOr(err, E_LABEL);
    __syncthreads();
    if (threadIdx.x == 0) {
        long long tot = 0;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) tot += part[w];
        *out = tot;
        const float den = divisor > 0.0 ? float(divisor) : float(tot);
        *kscale = den > 0.f ? __fdiv_rn(grad_scale, den) : 0.f;
    }
}

struct FinalizeArgs {
    uint32_t flags;
    float w_ce, w_z, w_dce, w_fkl, w_rkl, w_grpo, w_ent;
    double divisor;  // > 0: normaliser of the loss slots (a split batch)
};

// Sums the per-cluster partials in cluster order (fp64) and writes the
// sixteen scalars (means over valid rows, or loss sums over the caller's
// divisor; unselected slots 0).
// One warp per slot (blockDim = 32 * NACC): lane l sums clusters l, l + 32,
// ..., then a butterfly adds the 32 lane sums.  Assignment and order are fixed,
// so the result is bit-identical from call to call.
__global__ void __launch_bounds__(32 * NACC) finalize_kernel(const double* partials, int nclusters,
                                                             const long long* n_valid,
                                                             FinalizeArgs a, float* out) {
    __shared__ double tot[NACC];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row kernel has completed
    const int t = threadIdx.x >> 5, lane = threadIdx.x & 31;
    double s = 0.0;
    for (int c = lane; c < nclusters; c += 32) s += partials[size_t(c) * NACC + t];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) tot[t] = s;
    __syncthreads();
    if (threadIdx.x != 0) return;
    double o[16];
    for (int i = 0; i < 16; ++i) o[i] = 0.0;
    const double n = double(*n_valid);
    const double nl = a.divisor > 0.0 ? a.divisor : n;  // loss slots
    o[HEADLOSS_SLOT_N_VALID] = n;
    if (n > 0.0) {
        // one fp64 division per normaliser (each is slow on this GPU), then
        // products: the fp32 outputs see no difference
        const double rn = 1.0 / n, rnl = a.divisor > 0.0 ? 1.0 / nl : rn;
        const uint32_t f = a.flags;
        if (f & L_CE) o[HEADLOSS_SLOT_CE] = tot[A_CE] * rnl;
        if (f & L_Z) o[HEADLOSS_SLOT_Z] = tot[A_Z] * rnl;
        if (f & L_DIST_CE) o[HEADLOSS_SLOT_DIST_CE] = tot[A_DCE] * rnl;
        if (f & L_FKL) o[HEADLOSS_SLOT_FKL] = tot[A_FKL] * rnl;
        if (f & L_RKL) o[HEADLOSS_SLOT_RKL] = tot[A_RKL] * rnl;
        if (f & L_GRPO) o[HEADLOSS_SLOT_GRPO] = tot[A_GRPO] * rnl;
        if (f & L_GRPO_STATS) {
            o[HEADLOSS_SLOT_NEW_LOGPROB] = tot[A_LP] * rn;
            o[HEADLOSS_SLOT_RATIO] = tot[A_RATIO] * rn;
            o[HEADLOSS_SLOT_CLIP_FRAC] = tot[A_NCLIP] * rn;
            o[HEADLOSS_SLOT_KL_K3] = tot[A_KL3] * rn;
            const double am = tot[A_ADV] * rn;
            const double var = tot[A_ADV2] * rn - am * am;
            o[HEADLOSS_SLOT_ADV_MEAN] = am;
            o[HEADLOSS_SLOT_ADV_STD] = var > 0.0 ? sqrt(var) : 0.0;
            o[HEADLOSS_SLOT_N_CLIPPED] = tot[A_NCLIP];
        }
        if (f & L_ENTROPY) o[HEADLOSS_SLOT_ENTROPY] = tot[A_ENT] * rnl;
        double total = 0.0;
        if (f & L_CE) total += double(a.w_ce) * o[HEADLOSS_SLOT_CE];
        if (f & L_Z) total += double(a.w_z) * o[HEADLOSS_SLOT_Z];
        if (f & L_DIST_CE) total += double(a.w_dce) * o[HEADLOSS_SLOT_DIST_CE];
        if (f & L_FKL) total += double(a.w_fkl) * o[HEADLOSS_SLOT_FKL];
        if (f & L_RKL) total += double(a.w_rkl) * o[HEADLOSS_SLOT_RKL];
        if (f & L_GRPO) total += double(a.w_grpo) * o[HEADLOSS_SLOT_GRPO];
        if (f & L_ENTROPY) total += double(a.w_ent) * o[HEADLOSS_SLOT_ENTROPY];
        o[HEADLOSS_SLOT_TOTAL] = total;
    }
    for (int i = 0; i < 16; ++i) out[i] = float(o[i]);
}

}  // namespace hl

using namespace hl;

namespace {

constexpr uint32_t kAllFlags = 0xffu;
constexpr int kLaunchesPerCall = 3;

struct Plan {
    int64_t V = -1;
    int dtype = -1, feat = -1, inplace = -1;
    int kind = 0;  // HEADLOSS_KERNEL_RESIDENT or HEADLOSS_KERNEL_STREAM
    int C = 0, nbuf = 0, words = 0, smem = 0, ncl = 0, threads = 0, chunk_words = 0;
    int64_t L = 0;
    const void* kernel = nullptr;
};

}  // namespace

struct headloss {
    uint32_t flags;
    headloss_weights w;
    float T, eps, softcap, s;
    int device, num_sms, smem_optin;
    void* ws;
    double* partials;
    int partials_cap;  // clusters (resident) or CTAs (streaming)
    long long* n_valid;
    float* kscale;  // 8 bytes after n_valid
    int* err;
    headloss_plan_desc forced;  // zero fields: the planner decides
    Plan plan;                  // cache of the last plan
    std::mutex mu;
    unsigned long long wait_ns = 2000000000ull;  // limit of every in-kernel wait
    int64_t drop_row = -1;                       // fault-injection builds only
};

namespace {

int elem_size(int dtype) { return dtype == HEADLOSS_FP32 ? 4 : 2; }

int feature_set(const headloss* h) {
    int f = 0;
    if (h->flags & (L_DIST_CE | L_FKL | L_RKL)) f |= F_TEACH;
    if (h->flags & L_RKL) f |= F_RKL;
    if (h->flags & L_ENTROPY) f |= F_ENT;
    if (h->softcap > 0.f) f |= F_SOFTCAP;
    if (h->flags & L_DIST_CE) f |= F_DCE;
    if ((h->flags & L_ENTROPY) && h->w.entropy != 0.f) f |= F_ENTG;
    if ((f & F_TEACH) && h->T == 2.f) f |= F_T2;
    return f;
}

// fp32 rows in double-float arithmetic where fp32 pairs carry the precision:
// no teacher, no softcap, no entropy gradient term, and no accumulation (each
// term is good to ~2^-26 of itself, which an existing value of the opposite
// sign could leave exposed).
bool uses_df(int dtype, int feat) {
    return dtype == HEADLOSS_FP32 && !(feat & (F_ACC | F_TEACH | F_SOFTCAP | F_ENTG));
}

// The kernel of `kind` for `dtype` and the feature set `feat` (F_ACC selects
// the accumulating instantiation; the fp32 kernel reads the flag at run time).
const void* kernel_for(int kind, int dtype, int feat) {
    const bool df = uses_df(dtype, feat);
    const bool acc = (feat & F_ACC) != 0;
    feat &= ~F_ACC;
    if (kind == HEADLOSS_KERNEL_STREAM) {
        // L2 hints on the copies of teacher rows without softcap (measured:
        // distillation 2.77 -> 2.68 ms; with softcap, the all-in set, slower)
        if (!acc && (feat & F_TEACH) && !(feat & F_SOFTCAP)) feat |= F_L2P;
        // the T = 2 form: hinted bf16 instantiations without entropy only
        if (!((feat & F_L2P) && dtype == HEADLOSS_BF16 && !(feat & F_ENT))) feat &= ~F_T2;
        switch (dtype) {
            case HEADLOSS_BF16: return acc ? stream_kernel_bf16_acc(feat) : stream_kernel_bf16(feat);
            case HEADLOSS_FP16: return acc ? stream_kernel_fp16_acc(feat) : stream_kernel_fp16(feat);
            default: return nullptr;
        }
    }
    if (acc && dtype == HEADLOSS_BF16) return rows_kernel_bf16_acc(feat & F_BASE);
    if (acc && dtype == HEADLOSS_FP16) return rows_kernel_fp16_acc(feat & F_BASE);
    switch (dtype) {
        case HEADLOSS_BF16: return rows_kernel_bf16(feat & F_BASE);
        case HEADLOSS_FP16: return rows_kernel_fp16(feat & F_BASE);
        case HEADLOSS_FP32: return rows_kernel_fp32((feat & F_BASE) | (df ? int(F_DF) : 0));
        default: return nullptr;
    }
}

// Max co-resident clusters of `C` CTAs of `kernel` with `smem` bytes each.
int active_clusters(const void* kernel, int C, int threads, int smem, int num_sms, int* out) {
    if (C == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
            cudaSuccess)
            return HEADLOSS_ERR_CUDA;
        *out = per_sm * num_sms;
        return HEADLOSS_OK;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(C * num_sms, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(out, kernel, &cfg) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    return HEADLOSS_OK;
}

bool wants(int forced, int v) { return forced == 0 || forced == v; }

// Resident candidates: every cluster size C in 1..8, 512 or 256 threads,
// 1..4 row stages that fit in shared memory.
int resident_candidates(headloss* h, int64_t V, int dtype, int feat, Plan* cand, int* ncand) {
    const void* kernel = kernel_for(HEADLOSS_KERNEL_RESIDENT, dtype, feat);
    if (!kernel) return HEADLOSS_ERR_DTYPE;
    const int es = elem_size(dtype);
    const int epw = 16 / es;
    const int ops = (feat & F_TEACH) ? 2 : 1;
    const int acc_bytes = dtype == HEADLOSS_FP32 ? 8 : 4;
    const bool df = uses_df(dtype, feat);
    const int budget = h->smem_optin - smem_fixed_bytes(acc_bytes);
    // the attribute is a per-kernel cap shared by every handle: always the device maximum
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             h->smem_optin) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    static const int kThreads[] = {512, 256};
    for (int C = 1; C <= MAX_CLUSTER; ++C) {
        if (!wants(h->forced.cluster, C)) continue;
        int64_t L = (V + C - 1) / C;
        L = (L + epw - 1) / epw * epw;
        if (C > 1 && (C - 1) * L >= V && !h->forced.cluster) continue;  // an idle CTA
        const int64_t words = L / epw + 2;
        const int64_t stage = words * 16 * ops;
        // double-float: the low parts of the stored exponentials, bf16, one
        // set per CTA after the fixed area (16-byte aligned)
        const int64_t extra = df ? words * 8 + 16 : 0;
        const int64_t room = budget - extra;
        const int64_t max_nbuf =
            room / stage < MAX_RESIDENT_STAGES ? room / stage : MAX_RESIDENT_STAGES;
        for (int ti = 0; ti < 2; ++ti) {
            const int T = kThreads[ti];
            if (!wants(h->forced.threads, T)) continue;
            for (int64_t nbuf = 1; nbuf <= max_nbuf; ++nbuf) {
                if (!wants(h->forced.stages, int(nbuf))) continue;
                Plan pl;
                pl.kind = HEADLOSS_KERNEL_RESIDENT;
                pl.kernel = kernel;
                pl.C = C;
                pl.L = L;
                pl.words = int(words);
                pl.nbuf = int(nbuf);
                pl.threads = T;
                pl.smem = int(stage * nbuf + extra) + smem_fixed_bytes(acc_bytes);
                int ncl = 0;
                const int rc = active_clusters(kernel, C, T, pl.smem, h->num_sms, &ncl);
                if (rc) return rc;
                if (ncl > h->partials_cap) ncl = h->partials_cap;
                if (ncl < 1) continue;
                pl.ncl = ncl;
                cand[(*ncand)++] = pl;
            }
        }
    }
    return HEADLOSS_OK;
}

// Streaming candidates (16-bit logits with 16-byte aligned rows): 512 or 256
// threads, 1, 2 or 4 words per thread per chunk, 2..8 chunk slots.
int stream_candidates(headloss* h, int64_t V, int dtype, int feat, Plan* cand, int* ncand) {
    if (dtype == HEADLOSS_FP32 || (V * elem_size(dtype)) % 16 != 0) return HEADLOSS_OK;
    const void* kernel = kernel_for(HEADLOSS_KERNEL_STREAM, dtype, feat);
    if (!kernel) return HEADLOSS_ERR_DTYPE;
    const int ops = (feat & F_TEACH) ? 2 : 1;
    const int budget = h->smem_optin - smem_fixed_bytes(4);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             h->smem_optin) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    static const int kThreads[] = {512, 256};
    static const int kWords[] = {1, 2, 4};
    for (int ti = 0; ti < 2; ++ti) {
        const int T = kThreads[ti];
        if (!wants(h->forced.threads, T)) continue;
        for (int wi = 0; wi < 3; ++wi) {
            const int wpt = kWords[wi];
            if (!wants(h->forced.chunk_words, wpt)) continue;
            const int64_t CH = int64_t(wpt) * 8 * T;  // elements per chunk
            const int64_t slot = CH * 2 * ops;
            for (int S = 2; S <= MAX_STAGES; ++S) {
                if (!wants(h->forced.stages, S)) continue;
                if (slot * S > budget) break;
                Plan pl;
                pl.kind = HEADLOSS_KERNEL_STREAM;
                pl.kernel = kernel;
                pl.C = 1;
                pl.L = CH;
                pl.words = int(CH / 8);
                pl.nbuf = S;
                pl.threads = T;
                pl.chunk_words = wpt;
                pl.smem = int(slot * S) + smem_fixed_bytes(4);
                int n = 0;
                const int rc = active_clusters(kernel, 1, T, pl.smem, h->num_sms, &n);
                if (rc) return rc;
                if (n > h->partials_cap) n = h->partials_cap;
                if (n < 1) continue;
                pl.ncl = n;
                cand[(*ncand)++] = pl;
            }
        }
    }
    return HEADLOSS_OK;
}

// Resident rule (measured on GB300 across the five loss sets): many
// co-resident CTAs (two to four per SM, each holding one row slice) pay more
// than deep per-CTA staging -- one CTA's barriers, row merge and copy wait
// hide behind another's arithmetic.  So: a single-CTA cluster (no cluster
// exchange at all) if it fits at least two CTAs per SM; otherwise the plans
// within 20% of the most co-resident CTAs, and among them the smallest
// cluster, then one stage, then 256 threads (GRPO rows of 151936: 6-CTA
// clusters, 582 CTAs, 3.84 ms against 7-CTA clusters, 714 CTAs, 3.90 ms: a
// cluster's per-row barriers and merges grow with its size).
bool pick_resident(const headloss* h, const Plan* cand, int ncand, Plan* best) {
    int most = 0;
    for (int i = 0; i < ncand; ++i)
        if (cand[i].kind == HEADLOSS_KERNEL_RESIDENT && cand[i].ncl * cand[i].C > most)
            most = cand[i].ncl * cand[i].C;
    auto better = [](const Plan& a, const Plan& b) {
        if (a.C != b.C) return a.C < b.C;
        if (a.nbuf != b.nbuf) return a.nbuf < b.nbuf;
        return a.threads < b.threads;
    };
    Plan b;
    for (int i = 0; i < ncand; ++i) {
        const Plan& c = cand[i];
        if (c.kind == HEADLOSS_KERNEL_RESIDENT && c.C == 1 && c.ncl >= 2 * h->num_sms &&
            (b.C == 0 || better(c, b)))
            b = c;
    }
    if (b.C == 0)
        for (int i = 0; i < ncand; ++i) {
            const Plan& c = cand[i];
            if (c.kind == HEADLOSS_KERNEL_RESIDENT && double(c.ncl) * c.C >= 0.80 * most &&
                (b.C == 0 || better(c, b)))
                b = c;
        }
    if (b.C == 0) return false;
    *best = b;
    return true;
}

// Streaming rule (measured on GB300): the per-chunk bookkeeping (slot wait,
// shift check, release) is amortised over the chunk, so the largest chunk per
// thread wins; then the most co-resident CTAs (two CTAs of 256 threads beat
// one of 512: one CTA's row merge and barriers hide behind the other's
// arithmetic); then the most slots that still keep them co-resident (a
// deeper ring rides out DRAM latency: three slots beat two by ~1%).
// Except for teacher rows without softcap (`fewer_rows`): there one CTA of
// 512 threads per SM halves the rows in flight, so that with the gradient
// stores kept out of L2 a row's second read finds nearly all of it still
// there (DRAM bytes 1.34x -> 1.06x the minimum on the distillation set,
// 2.625 -> 2.602 ms); with softcap the arithmetic is heavier and two CTAs per
// SM still win (all-in 11.75 against 12.06 ms).
bool pick_stream(const headloss* h, const Plan* cand, int ncand, bool fewer_rows, Plan* best) {
    Plan b;
    double bscore = -1.0;
    for (int i = 0; i < ncand; ++i) {
        const Plan& c = cand[i];
        if (c.kind != HEADLOSS_KERNEL_STREAM) continue;
        const double score = c.chunk_words * 1e6 + (fewer_rows ? c.threads * 1e3 : 0.0) +
                             double(c.ncl) * 1e2 + c.nbuf;
        if (score > bscore) {
            b = c;
            bscore = score;
        }
    }
    if (bscore < 0) return false;
    (void)h;
    *best = b;
    return true;
}

// Chooses the kernel and its launch plan for rows of V elements of `dtype`.
// Measured on GB300 over the five loss sets: the streaming kernel wins when a
// row carries a teacher (twice the bytes and twice the exponentials per
// column, so a resident row needs a cluster of three or more CTAs and its
// per-row cluster barriers cost the most), and loses when the row is
// student-only (its second read, partly from DRAM, costs more than the
// resident kernel's barriers).  So: streaming for 16-bit rows with a teacher
// whose resident plan needs three or more CTAs per row; resident otherwise.
// A call whose gradient overwrites its logits (in place) always takes the
// resident kernel: it reads each row once into shared memory before any of
// the row's gradient is stored, while the streaming kernel reads the row a
// second time from global memory as it stores the gradient.  So does a call
// with a per-token coefficient (only the resident kernels apply one).
int make_plan(headloss* h, int64_t V, int dtype, Plan* out, int acc = 0, int inplace = 0) {
    const int feat = feature_set(h) | (acc ? int(F_ACC) : 0);
    if (h->plan.V == V && h->plan.dtype == dtype && h->plan.feat == feat &&
        h->plan.inplace == inplace) {
        *out = h->plan;
        return HEADLOSS_OK;
    }
    Plan cand[2 * MAX_CLUSTER * 2 * MAX_STAGES + 2 * 3 * MAX_STAGES];
    int ncand = 0;
    const int fk = inplace ? int(HEADLOSS_KERNEL_RESIDENT) : h->forced.kernel;
    int rc = HEADLOSS_OK;
    if (fk == 0 || fk == HEADLOSS_KERNEL_RESIDENT)
        rc = resident_candidates(h, V, dtype, feat, cand, &ncand);
    if (rc) return rc;
    if (fk == 0 || fk == HEADLOSS_KERNEL_STREAM) rc = stream_candidates(h, V, dtype, feat, cand, &ncand);
    if (rc) return rc;
    Plan res, str, best;
    const bool have_res = pick_resident(h, cand, ncand, &res);
    // the rows the hinted streaming instantiation takes (kernel_for)
    const bool fewer_rows = !acc && (feat & F_TEACH) && !(feat & F_SOFTCAP);
    const bool have_str = pick_stream(h, cand, ncand, fewer_rows, &str);
    if (fk == HEADLOSS_KERNEL_STREAM) {
        if (!have_str) return HEADLOSS_ERR_SIZE;
        best = str;
    } else if (fk == HEADLOSS_KERNEL_RESIDENT) {
        if (!have_res) return HEADLOSS_ERR_SIZE;
        best = res;
    } else if (have_str && (!have_res || (res.C >= 3 && (feat & F_TEACH)))) {
        best = str;
    } else if (have_res) {
        best = res;
    } else {
        return HEADLOSS_ERR_SIZE;
    }
    best.V = V;
    best.dtype = dtype;
    best.feat = feat;
    best.inplace = inplace;
    h->plan = best;
    *out = best;
    return HEADLOSS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int headloss_version(void) { return 1; }

int headloss_launches_per_call(void) { return kLaunchesPerCall; }

const char* headloss_strerror(int status) {
    switch (status) {
        case HEADLOSS_OK: return "ok";
        case HEADLOSS_ERR_ARG: return "invalid argument";
        case HEADLOSS_ERR_DTYPE: return "unsupported dtype";
        case HEADLOSS_ERR_ALIGN: return "logits, teacher or gradient base is not 16-byte aligned";
        case HEADLOSS_ERR_MISSING_INPUT: return "a selected loss is missing a required input";
        case HEADLOSS_ERR_CUDA: return "CUDA runtime error";
        case HEADLOSS_ERR_TIMEOUT: return "device: a bounded wait for a row copy gave up";
        case HEADLOSS_ERR_LABEL_RANGE: return "device: label >= V (row treated as masked)";
        case HEADLOSS_ERR_SIZE: return "vocabulary row too large for the on-chip plan";
        default: return "unknown status";
    }
}

int headloss_create(uint32_t flags, const headloss_weights* w, float temperature, float clip_eps,
                    float softcap, float logits_scale, headloss_t* out) {
    if (!out) return HEADLOSS_ERR_ARG;
    *out = nullptr;
    if (flags == 0 || (flags & ~kAllFlags)) return HEADLOSS_ERR_ARG;
    if (!(temperature > 0.f) || !isfinite(temperature)) return HEADLOSS_ERR_ARG;
    if (!(clip_eps >= 0.f) || !isfinite(clip_eps)) return HEADLOSS_ERR_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap)) return HEADLOSS_ERR_ARG;
    if (!(logits_scale > 0.f) || !isfinite(logits_scale)) return HEADLOSS_ERR_ARG;
    headloss_weights ww = {0.f, 0.f, 0.f, 0.f, 0.f, 1.f, 0.f, 1.f};
    ww.ce = 1.f;
    if (w) ww = *w;
    const float wl[8] = {ww.ce, ww.z, ww.dist_ce, ww.fkl, ww.rkl, ww.grpo, ww.entropy, ww.grad_scale};
    for (float v : wl)
        if (!isfinite(v)) return HEADLOSS_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    headloss* h = new (std::nothrow) headloss();
    if (!h) return HEADLOSS_ERR_ARG;
    h->flags = flags;
    h->w = ww;
    h->T = temperature;
    h->eps = clip_eps;
    h->softcap = softcap;
    h->s = logits_scale;
    h->device = dev;
    h->num_sms = sms;
    h->smem_optin = optin;
    h->partials_cap = 4 * sms;
    const size_t pbytes = size_t(h->partials_cap) * NACC * sizeof(double);
    if (cudaMalloc(&h->ws, pbytes + 256) != cudaSuccess) {
        delete h;
        return HEADLOSS_ERR_CUDA;
    }
    h->partials = static_cast<double*>(h->ws);
    h->n_valid = reinterpret_cast<long long*>(static_cast<char*>(h->ws) + pbytes);
    h->kscale = reinterpret_cast<float*>(static_cast<char*>(h->ws) + pbytes + 8);
    h->err = reinterpret_cast<int*>(static_cast<char*>(h->ws) + pbytes + 64);
    if (cudaMemset(h->ws, 0, pbytes + 256) != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return HEADLOSS_ERR_CUDA;
    }
    *out = h;
    return HEADLOSS_OK;
}

void headloss_destroy(headloss_t h) {
    if (!h) return;
    cudaFree(h->ws);
    delete h;
}

int headloss_force_plan(headloss_t h, const headloss_plan_desc* plan) {
    if (!h) return HEADLOSS_ERR_ARG;
    headloss_plan_desc d = {0, 0, 0, 0, 0};
    if (plan) d = *plan;
    if (d.kernel < 0 || d.kernel > HEADLOSS_KERNEL_STREAM) return HEADLOSS_ERR_ARG;
    if (d.cluster < 0 || d.cluster > MAX_CLUSTER) return HEADLOSS_ERR_ARG;
    if (d.stages < 0 || d.stages > MAX_STAGES) return HEADLOSS_ERR_ARG;
    if (!(d.threads == 0 || d.threads == 256 || d.threads == 512)) return HEADLOSS_ERR_ARG;
    if (!(d.chunk_words == 0 || d.chunk_words == 1 || d.chunk_words == 2 || d.chunk_words == 4))
        return HEADLOSS_ERR_ARG;
    std::lock_guard<std::mutex> g(h->mu);
    h->forced = d;
    h->plan = Plan();
    return HEADLOSS_OK;
}

int headloss_plan(headloss_t h, int64_t V, int dtype, headloss_plan_desc* plan, int* ctas,
                  int* smem_bytes) {
    if (!h || V < 1 || V >= (int64_t(1) << 31)) return HEADLOSS_ERR_ARG;
    if (dtype < 0 || dtype > 2) return HEADLOSS_ERR_DTYPE;
    std::lock_guard<std::mutex> g(h->mu);
    Plan pl;
    const int rc = make_plan(h, V, dtype, &pl);
    if (rc) return rc;
    if (plan) {
        plan->kernel = pl.kind;
        plan->cluster = pl.C;
        plan->stages = pl.nbuf;
        plan->threads = pl.threads;
        plan->chunk_words = pl.chunk_words;
    }
    if (ctas) *ctas = pl.ncl * pl.C;
    if (smem_bytes) *smem_bytes = pl.smem;
    return HEADLOSS_OK;
}

int headloss_forward_backward(headloss_t h, const void* logits, int64_t N, int64_t V, int dtype,
                              const int64_t* labels, const void* teacher_logits,
                              const float* old_logprobs, const float* advantages, void* grad_out,
                              float* scalars_out, headloss_stream_t stream) {
    return headloss_forward_backward_ext(h, logits, N, V, dtype, labels, teacher_logits,
                                         old_logprobs, advantages, grad_out, scalars_out,
                                         nullptr, stream);
}

// Host-side checks of a call (no device work): the argument, alignment and
// missing-input errors of headloss_forward_backward_ext, in its order.
static int check_call(const headloss* h, const void* logits, int64_t N, int64_t V, int dtype,
                      const int64_t* labels, const void* teacher_logits,
                      const float* old_logprobs, const float* advantages, const void* grad_out,
                      const float* scalars_out, const headloss_call_ext& x) {
    if (!h || !scalars_out || N < 0 || V < 1 || V >= (int64_t(1) << 31)) return HEADLOSS_ERR_ARG;
    if (!(x.divisor >= 0.0) || !isfinite(x.divisor)) return HEADLOSS_ERR_ARG;
    if (x.accumulate != 0 && x.accumulate != 1) return HEADLOSS_ERR_ARG;
    if (x.accumulate && !grad_out) return HEADLOSS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(x.new_logprobs) & 3u) ||
        (reinterpret_cast<uintptr_t>(x.row_loss) & 3u) ||
        (reinterpret_cast<uintptr_t>(x.token_coeff) & 3u))
        return HEADLOSS_ERR_ALIGN;
    if (N > 0 && !logits) return HEADLOSS_ERR_ARG;
    if (dtype < 0 || dtype > 2) return HEADLOSS_ERR_DTYPE;
    const uint32_t f = h->flags;
    if (N > 0) {  // an empty batch reads no input
        if ((f & (L_CE | L_GRPO | L_GRPO_STATS)) && !labels) return HEADLOSS_ERR_MISSING_INPUT;
        if ((f & (L_DIST_CE | L_FKL | L_RKL)) && !teacher_logits)
            return HEADLOSS_ERR_MISSING_INPUT;
        if ((f & (L_GRPO | L_GRPO_STATS)) && (!old_logprobs || !advantages))
            return HEADLOSS_ERR_MISSING_INPUT;
        if ((x.new_logprobs || x.token_coeff) && !labels) return HEADLOSS_ERR_MISSING_INPUT;
    }
    const bool teach = (f & (L_DIST_CE | L_FKL | L_RKL)) != 0;
    if (!aligned16(logits) || (teach && !aligned16(teacher_logits)) ||
        (grad_out && !aligned16(grad_out)))
        return HEADLOSS_ERR_ALIGN;
    if (teach && grad_out) {  // the gradient may alias the logits, never the teacher
        const char* g0 = static_cast<const char*>(grad_out);
        const char* t0 = static_cast<const char*>(teacher_logits);
        const int64_t bytes = N * V * elem_size(dtype);
        if (g0 < t0 + bytes && t0 < g0 + bytes) return HEADLOSS_ERR_ARG;
    }
    if (x.accumulate && N > 0) {  // accumulating into the logits themselves is refused
        const char* g0 = static_cast<const char*>(grad_out);
        const char* x0 = static_cast<const char*>(logits);
        const int64_t bytes = N * V * elem_size(dtype);
        if (g0 < x0 + bytes && x0 < g0 + bytes) return HEADLOSS_ERR_ARG;
    }
    return HEADLOSS_OK;
}

int headloss_forward_backward_ext(headloss_t h, const void* logits, int64_t N, int64_t V,
                                  int dtype, const int64_t* labels, const void* teacher_logits,
                                  const float* old_logprobs, const float* advantages,
                                  void* grad_out, float* scalars_out,
                                  const headloss_call_ext* ext, headloss_stream_t stream) {
    headloss_call_ext x = {nullptr, nullptr, 0, 0.0, nullptr};
    if (ext) x = *ext;
    {
        const int rc = check_call(h, logits, N, V, dtype, labels, teacher_logits, old_logprobs,
                                  advantages, grad_out, scalars_out, x);
        if (rc) return rc;
    }
    const uint32_t f = h->flags;
    const bool teach = (f & (L_DIST_CE | L_FKL | L_RKL)) != 0;
    std::lock_guard<std::mutex> g(h->mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    if (dev != h->device) return HEADLOSS_ERR_ARG;
    Plan pl;
    int inplace = 0;  // the gradient overlaps the logits
    if (grad_out && N > 0) {
        const char* g0 = static_cast<const char*>(grad_out);
        const char* x0 = static_cast<const char*>(logits);
        const int64_t bytes = N * V * elem_size(dtype);
        inplace = (g0 < x0 + bytes && x0 < g0 + bytes) ? 1 : 0;
    }
    // a per-token coefficient is applied by the resident kernels only
    const int rc = make_plan(h, V, dtype, &pl, x.accumulate, inplace || x.token_coeff ? 1 : 0);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    count_valid_kernel<<<1, 1024, 0, s>>>(labels, N, V, h->n_valid, h->err, h->w.grad_scale,
                                          x.divisor, h->kscale);

    int ncl = 0;
    if (N > 0) {
        ncl = int(N < pl.ncl ? N : pl.ncl);
        Params p;
        p.x = logits;
        p.t = teach ? teacher_logits : nullptr;
        p.g = grad_out;
        p.labels = labels;
        p.old_lp = (f & (L_GRPO | L_GRPO_STATS)) ? old_logprobs : nullptr;
        p.adv = (f & (L_GRPO | L_GRPO_STATS)) ? advantages : nullptr;
        p.N = N;
        p.V = V;
        p.L = pl.L;
        p.C = pl.C;
        p.nbuf = pl.nbuf;
        p.words = pl.words;
        p.flags = f;
        p.s = h->s;
        p.softcap = h->softcap;
        p.T = h->T;
        p.eps = h->eps;
        p.w_ce = h->w.ce;
        p.w_z = h->w.z;
        p.w_dce = h->w.dist_ce;
        p.w_fkl = h->w.fkl;
        p.w_rkl = h->w.rkl;
        p.w_grpo = h->w.grpo;
        p.w_ent = h->w.entropy;
        p.grad_scale = h->w.grad_scale;
        p.partials = h->partials;
        p.n_valid = h->n_valid;
        p.kscale = h->kscale;
        p.err = h->err;
        p.wait_ns = h->wait_ns;
        p.drop_row = h->drop_row;
        p.lp_out = x.new_logprobs;
        p.rl_out = x.row_loss;
        p.divisor = x.divisor;
        p.accumulate = x.accumulate;
        p.tok = x.token_coeff;

        // programmatic dependent launch: the row kernel's CTAs start while
        // the count kernel runs and wait for it before they read the count
        // (griddepcontrol.wait); the finalize kernel likewise after the row
        // kernel (measured: CE + z 0.206 -> 0.202 ms, the larger sets ~0.2%)
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = pl.C;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.gridDim = dim3(ncl * pl.C, 1, 1);
        cfg.blockDim = dim3(pl.threads, 1, 1);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = pl.C > 1 ? 2 : 1;
        void* args[] = {&p};
        if (cudaLaunchKernelExC(&cfg, pl.kernel, args) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    }
    FinalizeArgs fa;
    fa.flags = f;
    fa.w_ce = h->w.ce;
    fa.w_z = h->w.z;
    fa.w_dce = h->w.dist_ce;
    fa.w_fkl = h->w.fkl;
    fa.w_rkl = h->w.rkl;
    fa.w_grpo = h->w.grpo;
    fa.w_ent = h->w.entropy;
    fa.divisor = x.divisor;
    {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(1, 1, 1);
        cfg.blockDim = dim3(32 * NACC, 1, 1);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const double* pp = h->partials;
        int n = int(ncl);
        const long long* nvp = h->n_valid;
        void* args[] = {&pp, &n, &nvp, &fa, &scalars_out};
        if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&finalize_kernel), args) !=
            cudaSuccess)
            return HEADLOSS_ERR_CUDA;
    }
    return HEADLOSS_OK;
}

#ifdef HL_FAULT_INJECT
// Test builds only (never in libheadloss.so): skip the bulk copies of one
// row and shorten every in-kernel wait, so a test can watch a bounded wait
// give up and report HEADLOSS_ERR_TIMEOUT without hanging anything.
int headloss_test_inject(headloss_t h, int64_t drop_row, unsigned long long wait_ns) {
    if (!h) return HEADLOSS_ERR_ARG;
    h->drop_row = drop_row;
    h->wait_ns = wait_ns ? wait_ns : 2000000000ull;
    return HEADLOSS_OK;
}
#endif

int headloss_get_device_error(headloss_t h, headloss_stream_t stream, int* err) {
    if (!h || !err) return HEADLOSS_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    if (cudaMemcpy(&v, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    *err = (v & E_LABEL) ? HEADLOSS_ERR_LABEL_RANGE
                         : ((v & E_TIMEOUT) ? HEADLOSS_ERR_TIMEOUT : HEADLOSS_OK);
    return HEADLOSS_OK;
}

// The loss's gradient pass alone, from the per-tile row statistics of the
// LM-head GEMM (include/headloss.h documents the call).
int headloss_forward_backward_rowstats(headloss_t h, const void* logits, int64_t N, int64_t V,
                                       int dtype, const int64_t* labels,
                                       const void* teacher_logits, const float* old_logprobs,
                                       const float* advantages, const void* row_stats,
                                       const float* row_stats_t, const void* teacher_stats,
                                       void* grad_out, float* scalars_out,
                                       const headloss_call_ext* ext, headloss_stream_t stream) {
    headloss_call_ext x = {nullptr, nullptr, 0, 0.0, nullptr};
    if (ext) x = *ext;
    if (!h) return HEADLOSS_ERR_ARG;
    const uint32_t f = h->flags;
    // reverse KL's coefficient needs a cross sum before the gradient pass
    if (f & L_RKL) return HEADLOSS_ERR_ARG;
    const bool teach = (f & (L_DIST_CE | L_FKL)) != 0;
    {
        const int rc = check_call(h, logits, N, V, dtype, labels, teacher_logits, old_logprobs,
                                  advantages, grad_out, scalars_out, x);
        if (rc) return rc;
    }
    if (dtype != HEADLOSS_BF16) return HEADLOSS_ERR_DTYPE;
    if (V % 256) return HEADLOSS_ERR_ARG;
    if (N > 0 && !row_stats) return HEADLOSS_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(row_stats) & 15u) return HEADLOSS_ERR_ALIGN;
    if (teach && N > 0) {
        if (!teacher_stats) return HEADLOSS_ERR_MISSING_INPUT;
        if (h->T != 1.f && !row_stats_t) return HEADLOSS_ERR_MISSING_INPUT;
    }
    if ((reinterpret_cast<uintptr_t>(teacher_stats) & 15u) ||
        (reinterpret_cast<uintptr_t>(row_stats_t) & 3u))
        return HEADLOSS_ERR_ALIGN;
    std::lock_guard<std::mutex> g(h->mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    if (dev != h->device) return HEADLOSS_ERR_ARG;
    int feat = feature_set(h) & (F_TEACH | F_ENT | F_SOFTCAP | F_ENTG);
    const void* kernel = onepass_kernel_bf16(feat);
    if (!kernel) return HEADLOSS_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    count_valid_kernel<<<1, 1024, 0, s>>>(labels, N, V, h->n_valid, h->err, h->w.grad_scale,
                                          x.divisor, h->kscale);
    int grid = 0;
    if (N > 0) {
        // four warps per row (each a quarter of its words), eight warps per
        // CTA, as many CTAs as are resident together (two per SM: each
        // warp's copy ring is 12 KB)
        const int smem = onepass_smem_bytes();
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return HEADLOSS_ERR_CUDA;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, size_t(smem)) !=
                cudaSuccess ||
            per_sm < 1)
            return HEADLOSS_ERR_CUDA;
        const int64_t want = (4 * N + 7) / 8;
        const int64_t res = int64_t(per_sm) * h->num_sms;
        const int64_t cap = res < h->partials_cap ? res : h->partials_cap;
        grid = int(want < cap ? want : cap);
        Params p = {};
        p.x = logits;
        p.t = teach ? teacher_logits : nullptr;
        p.g = grad_out;
        p.labels = labels;
        p.old_lp = (f & (L_GRPO | L_GRPO_STATS)) ? old_logprobs : nullptr;
        p.adv = (f & (L_GRPO | L_GRPO_STATS)) ? advantages : nullptr;
        p.N = N;
        p.V = V;
        p.C = 1;
        p.flags = f;
        p.s = h->s;
        p.softcap = h->softcap;
        p.T = h->T;
        p.eps = h->eps;
        p.w_ce = h->w.ce;
        p.w_z = h->w.z;
        p.w_grpo = h->w.grpo;
        p.w_ent = h->w.entropy;
        p.w_dce = h->w.dist_ce;
        p.w_fkl = h->w.fkl;
        p.grad_scale = h->w.grad_scale;
        p.partials = h->partials;
        p.n_valid = h->n_valid;
        p.kscale = h->kscale;
        p.err = h->err;
        p.wait_ns = h->wait_ns;
        p.drop_row = -1;
        p.lp_out = x.new_logprobs;
        p.rl_out = x.row_loss;
        p.divisor = x.divisor;
        p.accumulate = x.accumulate;
        p.tok = x.token_coeff;
        int nt = int(V / 256);
        const void* rs = row_stats;
        const void* rsT = teach ? static_cast<const void*>(row_stats_t) : nullptr;
        const void* rst = teach ? teacher_stats : nullptr;
        void* args[] = {&p, &rs, &rsT, &rst, &nt};
        if (cudaLaunchKernel(kernel, dim3(grid), dim3(256), args, size_t(smem), s) !=
            cudaSuccess)
            return HEADLOSS_ERR_CUDA;
    }
    FinalizeArgs fa;
    fa.flags = f;
    fa.w_ce = h->w.ce;
    fa.w_z = h->w.z;
    fa.w_dce = h->w.dist_ce;
    fa.w_fkl = h->w.fkl;
    fa.w_rkl = 0.f;  // refused above
    fa.w_grpo = h->w.grpo;
    fa.w_ent = h->w.entropy;
    fa.divisor = x.divisor;
    finalize_kernel<<<1, 32 * NACC, 0, s>>>(h->partials, grid, h->n_valid, fa, scalars_out);
    if (cudaGetLastError() != cudaSuccess) return HEADLOSS_ERR_CUDA;
    return HEADLOSS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// headloss_forward_backward_noalloc: the same call for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they compute the
// loss: code running while a CUDA graph is being captured on its stream
// (allocation is not allowed there), code behind a framework memory pool that
// forbids raw device allocations, or a real-time loop that must not touch the
// allocator.  The handle-based entry point needs a workspace allocated by
// headloss_create; this one keeps that workspace in a fixed file-scope device
// array instead, so it allocates nothing, ever.
//
// The array holds NOALLOC_MAX_SLOTS partial-sum slots (one per launched
// cluster or CTA, 16 doubles each) plus the valid-row count and the error
// word: 1024 * 128 + 256 bytes = 131,328 bytes, present on every device that
// loads this library, for the life of the process.  A launch never uses more
// slots than that (the planner caps its grid there); a launch that would
// still need more is rejected with HEADLOSS_ERR_SIZE.
// ---------------------------------------------------------------------------
namespace {

constexpr int NOALLOC_MAX_SLOTS = 1024;
constexpr size_t NOALLOC_PARTIAL_BYTES = size_t(NOALLOC_MAX_SLOTS) * NACC * sizeof(double);
constexpr size_t NOALLOC_BYTES = NOALLOC_PARTIAL_BYTES + 256;
constexpr int NOALLOC_MAX_DEVICES = 64;

// Host code must not use this name as an address: it only identifies the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on device `dev` (the current device),
// resolved once per device.
int noalloc_scratch(int dev, void** out) {
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return HEADLOSS_ERR_ARG;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return HEADLOSS_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return HEADLOSS_OK;
}

}  // namespace

extern "C" int headloss_forward_backward_noalloc(
    uint32_t flags, const headloss_weights* w, float temperature, float clip_eps, float softcap,
    float logits_scale, const void* logits, int64_t N, int64_t V, int dtype,
    const int64_t* labels, const void* teacher_logits, const float* old_logprobs,
    const float* advantages, void* grad_out, float* scalars_out, headloss_stream_t stream) {
    // the same configuration checks as headloss_create
    if (flags == 0 || (flags & ~kAllFlags)) return HEADLOSS_ERR_ARG;
    if (!(temperature > 0.f) || !isfinite(temperature)) return HEADLOSS_ERR_ARG;
    if (!(clip_eps >= 0.f) || !isfinite(clip_eps)) return HEADLOSS_ERR_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap)) return HEADLOSS_ERR_ARG;
    if (!(logits_scale > 0.f) || !isfinite(logits_scale)) return HEADLOSS_ERR_ARG;
    headloss_weights ww = {1.f, 0.f, 0.f, 0.f, 0.f, 1.f, 0.f, 1.f};
    if (w) ww = *w;
    const float wl[8] = {ww.ce, ww.z, ww.dist_ce, ww.fkl, ww.rkl, ww.grpo, ww.entropy, ww.grad_scale};
    for (float v : wl)
        if (!isfinite(v)) return HEADLOSS_ERR_ARG;
    int dev = 0, sms = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HEADLOSS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    void* scratch = nullptr;
    const int rc = noalloc_scratch(dev, &scratch);
    if (rc) return rc;

    // a handle on the host stack whose workspace is the scratch array
    headloss h;
    h.flags = flags;
    h.w = ww;
    h.T = temperature;
    h.eps = clip_eps;
    h.softcap = softcap;
    h.s = logits_scale;
    h.device = dev;
    h.num_sms = sms;
    h.smem_optin = optin;
    h.ws = scratch;
    h.partials = static_cast<double*>(scratch);
    h.partials_cap = NOALLOC_MAX_SLOTS < 4 * sms ? NOALLOC_MAX_SLOTS : 4 * sms;
    h.n_valid = reinterpret_cast<long long*>(static_cast<char*>(scratch) + NOALLOC_PARTIAL_BYTES);
    h.kscale = reinterpret_cast<float*>(static_cast<char*>(scratch) + NOALLOC_PARTIAL_BYTES + 8);
    h.err = reinterpret_cast<int*>(static_cast<char*>(scratch) + NOALLOC_PARTIAL_BYTES + 64);
    h.forced = headloss_plan_desc{0, 0, 0, 0, 0};
    // the call's own argument checks first: a rejected call enqueues nothing
    {
        const headloss_call_ext none = {nullptr, nullptr, 0, 0.0, nullptr};
        const int crc = check_call(&h, logits, N, V, dtype, labels, teacher_logits, old_logprobs,
                                   advantages, grad_out, scalars_out, none);
        if (crc) return crc;
    }
    if (N > 0) {
        Plan pl;
        {
            std::lock_guard<std::mutex> g(h.mu);
            const int prc = make_plan(&h, V >= 1 && V < (int64_t(1) << 31) ? V : 1,
                                      dtype >= 0 && dtype <= 2 ? dtype : 1, &pl);
            if (prc == HEADLOSS_OK && pl.ncl > NOALLOC_MAX_SLOTS) return HEADLOSS_ERR_SIZE;
        }
    }
    // the previous call's error bits must not leak into this one
    if (cudaMemsetAsync(h.err, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    return headloss_forward_backward(&h, logits, N, V, dtype, labels, teacher_logits,
                                     old_logprobs, advantages, grad_out, scalars_out, stream);
}
