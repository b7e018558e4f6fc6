// hl_rows.cuh -- the fused head-loss row kernel (sm_103a).
//
// One thread-block cluster owns one vocabulary row at a time; each CTA of the
// cluster owns a contiguous column slice of that row.  Per row:
//
//   load       the CTA bulk-copies its student (and teacher) slice from HBM
//              into its own shared memory (cp.async.bulk, completion on an
//              mbarrier), several rows ahead of the one being computed;
//   stats      pass A: slice max of the raw logits (the softcap / scale
//              transform is monotonic, so max z = transform(max x));
//              pass B: exponent sums relative to the slice max;
//   merge      each CTA pushes its partial record into every peer's shared
//              memory (DSMEM), one cluster barrier, every CTA merges the
//              records in rank order (identical, deterministic result);
//   epilogue   per-row losses and the superposition coefficients;
//   gradient   pass C re-reads the slice from shared memory (never from HBM)
//              and writes the combined gradient once, cast to the logits dtype.
//
// HBM traffic per row is therefore the minimum: logits (+ teacher) read once,
// gradient written once.
//
// Source of the operation: Fast-LLM issue #507 (Proposed direction: one
// softmax, all scalars and the combined gradient in one pass); PR #549
// (Approach: fp32 accumulation, one cast; Loss coverage); PR #558 (Design:
// grad_j = prob_coeff * softmax_j - label_coeff * delta(j, label), extended
// here by teacher and reverse-KL terms).
//
// Statistics are kept in base 2: zs = z * log2(e), so every exponential is
// one exp2 and the logits scale folds into the same multiply.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "hl_df.cuh"
#include "hl_params.h"

namespace hl {

// ------------------------------------------------------------------ PTX ----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// The same copy with an L2 cache-eviction hint (a policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t addr, double v) {
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(addr), "d"(v) : "memory");
}

// Bounded wait on an mbarrier phase: gives up after `limit_ns` of wall time
// (~2 s in normal builds) and reports it, so a lost copy can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// ------------------------------------------------------------ math ----

__device__ __forceinline__ float ex2(float x) { return exp2f(x); }
__device__ __forceinline__ double ex2(double x) { return exp2(x); }
__device__ __forceinline__ float lg2(float x) { return log2f(x); }
__device__ __forceinline__ double lg2(double x) { return log2(x); }
__device__ __forceinline__ float ex(float x) { return expf(x); }
__device__ __forceinline__ double ex(double x) { return exp(x); }
__device__ __forceinline__ float tnh(float x) { return tanhf(x); }
__device__ __forceinline__ double tnh(double x) { return tanh(x); }
__device__ __forceinline__ float csh(float x) { return coshf(x); }
__device__ __forceinline__ double csh(double x) { return cosh(x); }
__device__ __forceinline__ float amax(float a, float b) { return fmaxf(a, b); }
// Uncontracted multiply / subtract: the statistics pass must reproduce the
// row maximum exactly (its shifted logit is exactly 0), which an FMA that
// fuses x * K - max would not.
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double mul_rn(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ double sub_rn(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ double amax(double a, double b) { return fmax(a, b); }

// ------------------------------------------------------------ dtypes ----

template <typename DT>
struct DTraits;

template <>
struct DTraits<__nv_bfloat16> {
    using acc = float;
    static constexpr int EPW = 8;  // elements per 16-byte word
    static constexpr int ES = 2;
    __device__ static void unpack(const uint4& w, float* v) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(u[i] << 16);
            v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float* g) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * i], g[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
    }
    __device__ static float to_acc(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_acc(float v) { return __float2bfloat16_rn(v); }
};

template <>
struct DTraits<__half> {
    using acc = float;
    static constexpr int EPW = 8;
    static constexpr int ES = 2;
    __device__ static void unpack(const uint4& w, float* v) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static uint4 pack(const float* g) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(g[2 * i], g[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
    }
    __device__ static float to_acc(__half v) { return __half2float(v); }
    __device__ static __half from_acc(float v) { return __float2half_rn(v); }
};

// fp32 logits: statistics and gradient in fp64 so the fp32 gradient is
// correctly rounded to within an ulp or two.
template <>
struct DTraits<float> {
    using acc = double;
    static constexpr int EPW = 4;
    static constexpr int ES = 4;
    __device__ static void unpack(const uint4& w, double* v) {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
    __device__ static uint4 pack(const double* g) {
        return make_uint4(__float_as_uint(__double2float_rn(g[0])),
                          __float_as_uint(__double2float_rn(g[1])),
                          __float_as_uint(__double2float_rn(g[2])),
                          __float_as_uint(__double2float_rn(g[3])));
    }
    __device__ static double to_acc(float v) { return v; }
    __device__ static float from_acc(double v) { return __double2float_rn(v); }
};

// Shared-memory bytes beyond the stage buffers (mbarriers, exchange records,
// reduction scratch, row coefficients), for an accumulator of `acc_bytes`.
__host__ __device__ constexpr int smem_fixed_bytes(int acc_bytes) {
    // the last 32 words: a row's coefficients, then its losses waiting to be summed
    return 8 * MAX_STAGES + 8 * NACC +
           acc_bytes * (2 * MAX_CLUSTER * NREC + NWARPS * NREC + 2 * NWARPS + 32) +
           4 * MAX_STAGES;
}

// ---------------------------------------------------------- reductions ----

// Block reductions over the CTA's nwarps = blockDim.x / 32 (<= NWARPS) warps;
// the result is left in every lane of warp 0.
template <typename A, int NV>
__device__ __forceinline__ void block_sum(A (&v)[NV], A* red, int lane, int warp) {
    const int nwarps = int(blockDim.x >> 5);
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < NV; ++i) red[warp * NV + i] = v[i];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = lane < nwarps ? red[lane * NV + i] : A(0);
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
}

template <typename A, int NV>
__device__ __forceinline__ void block_max(A (&v)[NV], A* red, int lane, int warp) {
    const int nwarps = int(blockDim.x >> 5);
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = amax(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < NV; ++i) red[warp * NV + i] = v[i];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = lane < nwarps ? red[lane * NV + i] : A(-CUDART_INF);
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i)
                v[i] = amax(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
    }
}

// ------------------------------------------------------- row epilogue ----

// Row coefficients broadcast through shared memory.
enum Coef { K_LSE2, K_LSET2, K_LSQ2, K_PC, K_PS, K_TC, K_TS, K_QC, K_BC, NCOEF };

// Merges the C partial records (rank order), derives the row's losses,
// accumulates them (rank 0 only) and writes the gradient coefficients.
// Runs on one thread.  DFX (fp64 rows of the double-float kernel): its
// exponentials, logarithm and reciprocals through fp32 operations with
// fp64 corrections (hl_df.cuh) instead of fp64 library calls, which are slow
// on GB300; errors stay relative to the quantities that may cancel (the
// largest record's weight is exactly 1, log2 S near S = 1 is small).
template <typename A, bool TEACH, bool RKL, bool ENT, bool CAP, bool DFX = false>
__device__ void row_epilogue(const Params& p, const A* recs, int C, bool accumulate,
                             float old_lp, float adv, double* acc, A* coef, int64_t row) {
    static_assert(!DFX || (sizeof(A) == 8 && !TEACH && !CAP), "double-float epilogue");
    auto ex2_ = [](A v) -> A {
        if constexpr (DFX) return A(df_exp2d(double(v)));
        else return ex2(v);
    };
    const A LN2 = A(0.6931471805599453);
    const A invT = A(1) / A(p.T);
    A M = A(-CUDART_INF), Mu = A(-CUDART_INF);
    for (int k = 0; k < C; ++k) {
        const A* r = recs + k * NREC;
        if (r[R_S] > A(0)) {
            M = amax(M, r[R_ZM]);
            if (TEACH) Mu = amax(Mu, r[R_UM]);
        }
    }
    A S = 0, E = 0, ST = 0, Sq = 0, Eq = 0, Xp = 0, Y = 0, zy = 0;
    for (int k = 0; k < C; ++k) {
        const A* r = recs + k * NREC;
        if (r[R_HASY] > A(0)) zy = r[R_ZY];
        if (!(r[R_S] > A(0))) continue;
        const A d = r[R_ZM] - M;
        const A al = ex2_(d);
        S += al * r[R_S];
        if (ENT) E += al * (r[R_E] + d * r[R_S]);
        if (TEACH) {
            const A dT = d * invT;
            const A alT = ex2(dT);
            const A du = r[R_UM] - Mu;
            const A be = ex2(du);
            ST += alT * r[R_ST];
            Sq += be * r[R_SQ];
            Eq += be * (r[R_EQ] + du * r[R_SQ]);
            Xp += be * (r[R_XP] + (du - dT) * r[R_SQ]);
            if (RKL) Y += alT * (r[R_Y] - (du - dT) * r[R_ST]);
        }
    }
    const uint32_t f = p.flags;
    A lS;
    if constexpr (DFX) lS = A(df_log2d(double(S)));
    else lS = lg2(S);
    const A lse2 = M + lS;
    const A lse = lse2 * LN2;
    const double nv = p.divisor > 0.0 ? p.divisor : double(*p.n_valid);
    double k;
    if constexpr (DFX) k = double(p.grad_scale) * df_recipd(nv);
    else k = double(p.grad_scale) / nv;
    A H = 0, lST = 0, lSq = 0, dce = 0, fkl = 0, rkl = 0;
    if constexpr (DFX) {
        if (ENT) H = LN2 * (lS - E * A(df_recipd(double(S))));
    } else {
        if (ENT) H = LN2 * (lS - E / S);
    }
    if (TEACH) {
        lST = lg2(ST);
        lSq = lg2(Sq);
        fkl = LN2 * (Xp / Sq - lSq + lST);
        dce = LN2 * (Xp / Sq + lST - Eq / Sq);
        if (RKL) rkl = LN2 * (Y / ST - lST + lSq);
    }
    A pc = 0, ps = 0, tc = 0, ts = 0, qc = 0, bc = 0;
    const A kk = A(k);
    if (f & L_CE) {
        pc += kk * A(p.w_ce);
        bc += kk * A(p.w_ce);
    }
    if (f & L_Z) pc += kk * A(p.w_z) * A(2) * lse;
    A lp = 0, rho = 0, grpo = 0, kl3 = 0;
    bool clipped = false;
    if (f & (L_GRPO | L_GRPO_STATS)) {
        const A eps = A(p.eps);
        lp = (zy - lse2) * LN2;
        const A lr = lp - A(old_lp);
        if constexpr (DFX) rho = A(df_exp2d(double(lr) * (1.0 / DF_LN2)));
        else rho = ex(lr);
        A rho_c = rho < A(1) - eps ? A(1) - eps : rho;
        rho_c = rho_c > A(1) + eps ? A(1) + eps : rho_c;
        const A unc = rho * A(adv), clp = rho_c * A(adv);
        const A obj = unc < clp ? unc : clp;
        const bool act = unc <= clp || (rho >= A(1) - eps && rho <= A(1) + eps);
        grpo = -obj;
        kl3 = rho - A(1) - lr;
        clipped = fabs(double(rho) - 1.0) > double(eps);
        if ((f & L_GRPO) && act) {
            const A gco = kk * A(p.w_grpo) * A(adv) * rho;
            pc += gco;
            bc += gco;
        }
    }
    if (ENT && (f & L_ENTROPY)) {
        const A ec = kk * A(p.w_ent);
        pc -= ec * H;
        ps = -ec * LN2;
    }
    if (TEACH) {
        A dc = 0;
        if (f & L_DIST_CE) dc += A(p.w_dce);
        if (f & L_FKL) dc += A(p.w_fkl);
        dc *= kk * invT;
        tc += dc;
        qc -= dc;
        if (RKL && (f & L_RKL)) {
            const A rc = kk * invT * A(p.w_rkl);
            tc -= rc * rkl;
            ts = rc * LN2;
        }
    }
    if (!CAP) {  // dz/dx = s: fold the chain rule into the coefficients
        const A s = A(p.s);
        pc *= s;
        ps *= s;
        tc *= s;
        ts *= s;
        qc *= s;
        bc *= s;
    }
    coef[K_LSE2] = lse2;
    coef[K_LSET2] = TEACH ? M * invT + lST : A(0);
    coef[K_LSQ2] = TEACH ? Mu + lSq : A(0);
    coef[K_PC] = pc;
    coef[K_PS] = ps;
    coef[K_TC] = tc;
    coef[K_TS] = ts;
    coef[K_QC] = qc;
    coef[K_BC] = bc;
    if (accumulate) {
        acc[A_NVALID] += 1.0;
        if (f & L_CE) acc[A_CE] += double((lse2 - zy) * LN2);
        if (f & L_Z) acc[A_Z] += double(lse) * double(lse);
        if (f & L_DIST_CE) acc[A_DCE] += double(dce);
        if (f & L_FKL) acc[A_FKL] += double(fkl);
        if (f & L_RKL) acc[A_RKL] += double(rkl);
        if (f & L_GRPO) acc[A_GRPO] += double(grpo);
        if (f & L_GRPO_STATS) {
            acc[A_LP] += double(lp);
            acc[A_RATIO] += double(rho);
            acc[A_KL3] += double(kl3);
            acc[A_ADV] += double(adv);
            acc[A_ADV2] += double(adv) * double(adv);
            acc[A_NCLIP] += clipped ? 1.0 : 0.0;
        }
        if (f & L_ENTROPY) acc[A_ENT] += double(H);
        // per-token outputs
        if (p.lp_out) p.lp_out[row] = float((zy - lse2) * LN2);
        if (p.rl_out) {
            double t = 0.0;
            if (f & L_CE) t += double(p.w_ce) * double((lse2 - zy) * LN2);
            if (f & L_Z) t += double(p.w_z) * double(lse) * double(lse);
            if (f & L_DIST_CE) t += double(p.w_dce) * double(dce);
            if (f & L_FKL) t += double(p.w_fkl) * double(fkl);
            if (f & L_RKL) t += double(p.w_rkl) * double(rkl);
            if (f & L_GRPO) t += double(p.w_grpo) * double(grpo);
            if (f & L_ENTROPY) t += double(p.w_ent) * double(H);
            p.rl_out[row] = float(t);
        }
    }
}

}  // namespace hl
