// hl_rows_kernel.cuh -- the persistent cluster-per-row kernel (see hl_rows.cuh
// for the row pipeline and the sources it follows).
#pragma once
#include "hl_df.cuh"
#include "hl_rows.cuh"

namespace hl {

template <typename DT, int FEAT>
__global__ void __launch_bounds__(THREADS, 1) rows_kernel(const __grid_constant__ Params p) {
    using Tr = DTraits<DT>;
    using A = typename Tr::acc;
    constexpr int EPW = Tr::EPW;
    constexpr int ES = Tr::ES;
    constexpr bool TEACH = (FEAT & F_TEACH) != 0;
    constexpr bool RKL = (FEAT & F_RKL) != 0;
    constexpr bool ENT = (FEAT & F_ENT) != 0;
    constexpr bool CAP = (FEAT & F_SOFTCAP) != 0;
    constexpr int OPS = TEACH ? 2 : 1;
    // double-float element arithmetic (fp32 logits, no teacher, no softcap)
    constexpr bool DFM = (FEAT & F_DF) != 0;
    static_assert(!DFM || (sizeof(DT) == 4 && !TEACH && !CAP), "double-float feature set");

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = int(blockDim.x);
    const int W = p.words;
    const uint32_t opbytes = uint32_t(W) * 16u;
    const uint32_t stage_bytes = opbytes * OPS;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(stage_bytes) * p.nbuf);
    double* acc = reinterpret_cast<double*>(bars + MAX_STAGES);  // [NACC], thread 0 of rank 0
    A* xch = reinterpret_cast<A*>(acc + NACC);          // [2][MAX_CLUSTER][NREC]
    A* red = xch + 2 * MAX_CLUSTER * NREC;              // [NWARPS][NREC]
    A* coef = red + NWARPS * NREC;                      // [16]
    // double-float path: coef[13] the slice's raw maximum, coef[12] the label
    // logit (its shared-memory copy is overwritten by 2^d); the low parts of
    // the stored 2^d, as bf16, after the fixed area
    constexpr int DF_VMAX = 13, DF_VY = 12;
    float* const df_vy = reinterpret_cast<float*>(coef + DF_VY);  // fp32: no conversion per element
    __nv_bfloat16* elb = reinterpret_cast<__nv_bfloat16*>(
        smem + ((size_t(stage_bytes) * p.nbuf + smem_fixed_bytes(sizeof(A)) + 15) & ~size_t(15)));

    const int C = p.C;
    uint32_t rank, cid, ncl;
    if (C > 1) {
        rank = cluster_ctarank();
        cid = cluster_id_x();
        ncl = ncluster_x();
    } else {
        rank = 0;
        cid = blockIdx.x;
        ncl = gridDim.x;
    }
    const int64_t N = p.N, V = p.V;
    const int64_t col0 = int64_t(rank) * p.L;
    const int64_t col1 = col0 + p.L < V ? col0 + p.L : V;
    const DT* __restrict__ xg = static_cast<const DT*>(p.x);
    const DT* __restrict__ tg = static_cast<const DT*>(p.t);
    DT* gg = static_cast<DT*>(p.g);

    const A LOG2E = A(1.4426950408889634);
    const A s = A(p.s);
    const A K = s * LOG2E;                                 // zs = x * K (no softcap)
    const A invc = CAP ? A(1) / A(p.softcap) : A(0);
    const A Kc = CAP ? s * A(p.softcap) * LOG2E : A(0);    // zs = tanh(x / c) * Kc
    const A invT = A(1) / A(p.T);
    const A KT = LOG2E * invT;                             // us = t * KT

    auto zs_of = [&](A v) -> A { return CAP ? mul_rn(tnh(v * invc), Kc) : mul_rn(v, K); };
    // double-float split of an fp64 value (hi = its rounding, lo = the rest)
    auto split = [](double v) -> DF {
        const float h = float(v);
        return {h, float(v - double(h))};
    };
    const DF Kd = split(double(K));

    asm volatile("griddepcontrol.wait;" ::: "memory");  // the count kernel has completed
    if (tid == 0) {
        for (int b = 0; b < p.nbuf; ++b) mbar_init(smem_addr(&bars[b]), 1);
        fence_mbar_init();
        for (int i = 0; i < NACC; ++i) acc[i] = 0.0;
    }
    __syncthreads();
    if (C > 1) cluster_barrier();  // every peer has started before any DSMEM store

    // Producer (thread 0): start the copies of local iteration `it` into its stage.
    auto issue = [&](int it) {
        const int64_t r = int64_t(cid) + int64_t(it) * ncl;
        if (r >= N) return;
        const int st = it % p.nbuf;
        const uint32_t bar = smem_addr(&bars[st]);
        const int64_t e0 = r * V + col0, e1 = r * V + col1;
        int64_t f0 = (e0 + EPW - 1) / EPW * EPW, f1 = e1 / EPW * EPW;
        const uint32_t bytes = (e1 > e0 && f1 > f0) ? uint32_t((f1 - f0) * ES) : 0u;
        fence_proxy_async();  // order earlier generic stores to this stage before the copy
        mbar_arrive_expect_tx(bar, bytes * OPS);
#ifdef HL_FAULT_INJECT
        if (r == p.drop_row) return;  // the copy never comes: the wait must give up
#endif
        if (bytes) {
            const uint32_t dst = smem_addr(smem + size_t(st) * stage_bytes) +
                                 uint32_t((f0 / EPW - e0 / EPW) * 16);
            bulk_g2s(dst, xg + f0, bytes, bar);
            if (TEACH) bulk_g2s(dst + opbytes, tg + f0, bytes, bar);
        }
    };
    if (tid == 0)
        for (int it = 0; it < p.nbuf; ++it) issue(it);

    const bool has_labels = p.labels != nullptr;
    const bool need_side = (p.flags & (L_GRPO | L_GRPO_STATS)) != 0;
    int xc = 0;             // exchanges done (parity of the exchange buffer)
    uint32_t lost = 0, lost_par = 0;  // stages (and phase parities) whose wait gave up

    // Side inputs of the next row are loaded one iteration ahead.
    int64_t y_next = 0;
    float o_next = 0.f, a_next = 0.f;
    if (int64_t(cid) < N) {
        if (has_labels) y_next = p.labels[cid];
        if (need_side) {
            o_next = p.old_lp[cid];
            a_next = p.adv[cid];
        }
    }

    for (int it = 0;; ++it) {
        const int64_t r = int64_t(cid) + int64_t(it) * ncl;
        if (r >= N) break;
        const int64_t y = y_next;
        const float old_lp = o_next, adv = a_next;
        {
            const int64_t rn = r + ncl;
            if (rn < N) {
                if (has_labels) y_next = p.labels[rn];
                if (need_side) {
                    o_next = p.old_lp[rn];
                    a_next = p.adv[rn];
                }
            }
        }
        const bool valid = !has_labels || (y >= 0 && y < V);
        if (has_labels && y >= V && rank == 0 && tid == 0) atomicOr(p.err, E_LABEL);

        const int st = it % p.nbuf;
        const uint32_t par = uint32_t(it / p.nbuf) & 1u;
        if (!mbar_wait_bounded(smem_addr(&bars[st]), par, p.wait_ns)) {
            lost |= 1u << st;
            lost_par = (lost_par & ~(1u << st)) | (par << st);
            if (tid == 0) atomicOr(p.err, E_TIMEOUT);
        }
        unsigned char* xs_b = smem + size_t(st) * stage_bytes;
        DT* xs = reinterpret_cast<DT*>(xs_b);
        DT* ts = reinterpret_cast<DT*>(xs_b + opbytes);

        const int64_t e0 = r * V + col0, e1 = r * V + col1;
        const bool nonempty = e1 > e0;
        const int64_t wf = e0 / EPW;
        const int nw = nonempty ? int((e1 + EPW - 1) / EPW - wf) : 0;

        if (valid && nonempty) {
            // Elements of partial 16-byte words at the slice ends (rows whose
            // byte length is not a multiple of 16) come in with plain loads.
            const int64_t f0 = (e0 + EPW - 1) / EPW * EPW, f1 = e1 / EPW * EPW;
            const int64_t head_end = e1 < f0 ? e1 : f0;
            const int64_t tail_start = f1 > head_end ? f1 : head_end;
            const int nh = int(head_end - e0), nt = int(e1 - tail_start);
            if (nh + nt > 0) {
                if (tid < nh + nt) {
                    const int64_t e = tid < nh ? e0 + tid : tail_start + (tid - nh);
                    xs[e - wf * EPW] = xg[e];
                    if (TEACH) ts[e - wf * EPW] = tg[e];
                }
                __syncthreads();
            }
        }

        if (valid) {
            // ---- pass A: slice max of raw student / teacher logits ----
            A mx[2] = {A(-CUDART_INF), A(-CUDART_INF)};
            if constexpr (DFM) {
                // fp32 compares (exact), one fp32 block maximum
                float m1[1] = {-CUDART_INF_F};
                for (int w = tid; w < nw; w += nthr) {
                    const int64_t eb = (wf + w) * EPW;
                    const bool full = eb >= e0 && eb + EPW <= e1;
                    const float4 q4 = *reinterpret_cast<const float4*>(xs_b + size_t(w) * 16);
                    const float vv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int i = 0; i < EPW; ++i)
                        if (full || (eb + i >= e0 && eb + i < e1)) m1[0] = fmaxf(m1[0], vv[i]);
                }
                block_max<float, 1>(m1, reinterpret_cast<float*>(red), lane, warp);
                mx[0] = A(m1[0]);
            } else {
            for (int w = tid; w < nw; w += nthr) {
                const int64_t eb = (wf + w) * EPW;
                const bool full = eb >= e0 && eb + EPW <= e1;
                A v[EPW];
                Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + size_t(w) * 16), v);
#pragma unroll
                for (int i = 0; i < EPW; ++i)
                    if (full || (eb + i >= e0 && eb + i < e1)) mx[0] = amax(mx[0], v[i]);
                if (TEACH) {
                    Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + opbytes + size_t(w) * 16), v);
#pragma unroll
                    for (int i = 0; i < EPW; ++i)
                        if (full || (eb + i >= e0 && eb + i < e1)) mx[1] = amax(mx[1], v[i]);
                }
            }
            block_max<A, 2>(mx, red, lane, warp);
            }
            if (tid == 0) {
                coef[0] = nonempty ? zs_of(mx[0]) : A(-CUDART_INF);
                coef[1] = (TEACH && nonempty) ? mul_rn(mx[1], KT) : A(-CUDART_INF);
                if (DFM) coef[DF_VMAX] = mx[0];  // the raw maximum, for the double-float shift
            }
            __syncthreads();
            const A zm = coef[0], um = coef[1];

            // ---- pass B: exponent sums relative to the slice max ----
            // S = sum 2^d, E = sum 2^d d (d = zs - zm); ST = sum 2^(d/T);
            // Sq = sum 2^du, Eq = sum 2^du du (du = us - um);
            // Xp = sum 2^du (du - d/T);  Y = -sum 2^(d/T) (du - d/T).
            A sm[7] = {A(0), A(0), A(0), A(0), A(0), A(0), A(0)};
            if constexpr (DFM) {
                // S and E in double-float per thread: each term 2^d from
                // d = v K - v_max K formed to ~2^-48 (and exactly 0 at the
                // maximum, whose product is formed the same way: a one-column
                // row's CE is then exactly 0), summed by two-sums; terms below
                // 2^-126 (beside the maximum's 1) are dropped.  The shift
                // differs from the record's fp64 zm by ~2^-48 |zm|.  Each
                // 2^d, times 2^64, replaces its logit in shared memory (high
                // part; the low part as bf16 beside) for the gradient pass,
                // which then only scales it; the label logit is kept apart.
                const float vmax = float(coef[DF_VMAX]);
                DF Zd = df_two_prod(vmax, Kd.h);
                Zd.l = __fmaf_rn(vmax, Kd.l, Zd.l);
                const bool keep = gg != nullptr && !p.accumulate;
                const int64_t eyl = (has_labels && y >= col0 && y < col1) ? r * V + y : -1;
                float Sh = 0.f, Sl = 0.f, Eh = 0.f, El = 0.f;
                for (int w = tid; w < nw; w += nthr) {
                    const int64_t eb = (wf + w) * EPW;
                    const bool full = eb >= e0 && eb + EPW <= e1;
                    const float4 q4 = *reinterpret_cast<const float4*>(xs_b + size_t(w) * 16);
                    const float vv[4] = {q4.x, q4.y, q4.z, q4.w};
                    float kh[4], kl[4];
#pragma unroll
                    for (int i = 0; i < EPW; ++i) {
                        const bool in = full || (eb + i >= e0 && eb + i < e1);
                        if (eb + i == eyl) *df_vy = vv[i];
                        const DF d = df_scaled_minus(vv[i], Kd, Zd);
                        int n;
                        const DF e = df_exp2(d, n);
                        const bool big = n + 64 >= -126;  // 2^d 2^64 normal
                        const float s64 = big ? df_pow2i(n + 64) : 0.f;
                        kh[i] = __fmul_rn(e.h, s64);
                        kl[i] = __fmul_rn(e.l, s64);
                        if (!in || n < -126) continue;
                        const float sc = df_pow2i(n);
                        const float eh = __fmul_rn(e.h, sc), el = __fmul_rn(e.l, sc);
                        const DF s2 = df_two_sum(Sh, eh);
                        Sh = s2.h;
                        Sl = __fadd_rn(Sl, __fadd_rn(s2.l, el));
                        if (ENT) {
                            DF pe = df_two_prod(eh, d.h);
                            pe.l = __fmaf_rn(eh, d.l, __fmaf_rn(el, d.h, pe.l));
                            const DF e2 = df_two_sum(Eh, pe.h);
                            Eh = e2.h;
                            El = __fadd_rn(El, __fadd_rn(e2.l, pe.l));
                        }
                    }
                    if (keep) {
                        *reinterpret_cast<float4*>(xs_b + size_t(w) * 16) =
                            make_float4(kh[0], kh[1], kh[2], kh[3]);
                        __nv_bfloat162 l01 = __floats2bfloat162_rn(kl[0], kl[1]);
                        __nv_bfloat162 l23 = __floats2bfloat162_rn(kl[2], kl[3]);
                        *reinterpret_cast<uint2*>(elb + size_t(w) * 4) =
                            make_uint2(*reinterpret_cast<uint32_t*>(&l01),
                                       *reinterpret_cast<uint32_t*>(&l23));
                    }
                }
                // block sums in double-float (fp32 shuffles and two-sums),
                // converted to fp64 once, by warp 0
                auto add_df = [](float& h, float& l, float oh, float ol) {
                    const DF t = df_two_sum(h, oh);
                    h = t.h;
                    l = __fadd_rn(l, __fadd_rn(t.l, ol));
                };
                float* rf = reinterpret_cast<float*>(red);
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    add_df(Sh, Sl, __shfl_xor_sync(0xffffffffu, Sh, o),
                           __shfl_xor_sync(0xffffffffu, Sl, o));
                    if (ENT)
                        add_df(Eh, El, __shfl_xor_sync(0xffffffffu, Eh, o),
                               __shfl_xor_sync(0xffffffffu, El, o));
                }
                if (lane == 0) {
                    rf[4 * warp] = Sh;
                    rf[4 * warp + 1] = Sl;
                    rf[4 * warp + 2] = Eh;
                    rf[4 * warp + 3] = El;
                }
                __syncthreads();
                if (warp == 0) {
                    const int nwarps = nthr >> 5;
                    Sh = lane < nwarps ? rf[4 * lane] : 0.f;
                    Sl = lane < nwarps ? rf[4 * lane + 1] : 0.f;
                    Eh = lane < nwarps ? rf[4 * lane + 2] : 0.f;
                    El = lane < nwarps ? rf[4 * lane + 3] : 0.f;
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        add_df(Sh, Sl, __shfl_xor_sync(0xffffffffu, Sh, o),
                               __shfl_xor_sync(0xffffffffu, Sl, o));
                        if (ENT)
                            add_df(Eh, El, __shfl_xor_sync(0xffffffffu, Eh, o),
                                   __shfl_xor_sync(0xffffffffu, El, o));
                    }
                    sm[0] = double(Sh) + double(Sl);
                    if (ENT) sm[1] = double(Eh) + double(El);
                }
            } else {
            for (int w = tid; w < nw; w += nthr) {
                const int64_t eb = (wf + w) * EPW;
                const bool full = eb >= e0 && eb + EPW <= e1;
                A v[EPW], u[EPW];
                Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + size_t(w) * 16), v);
                if (TEACH)
                    Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + opbytes + size_t(w) * 16), u);
#pragma unroll
                for (int i = 0; i < EPW; ++i) {
                    if (!(full || (eb + i >= e0 && eb + i < e1))) continue;
                    const A d = sub_rn(zs_of(v[i]), zm);
                    const A e = ex2(d);
                    sm[0] += e;
                    if (ENT) sm[1] += e * d;
                    if (TEACH) {
                        const A dT = d * invT;
                        const A eT = ex2(dT);
                        const A du = sub_rn(mul_rn(u[i], KT), um);
                        const A eq = ex2(du);
                        const A wd = du - dT;
                        sm[2] += eT;
                        sm[3] += eq;
                        sm[4] += eq * du;
                        sm[5] += eq * wd;
                        if (RKL) sm[6] -= eT * wd;
                    }
                }
            }
            block_sum<A, 7>(sm, red, lane, warp);
            }
            A* myrec = xch + ((xc & 1) * MAX_CLUSTER + rank) * NREC;
            if (tid == 0) {
                A rec[NREC];
                rec[R_ZM] = zm;
                rec[R_UM] = um;
                rec[R_S] = sm[0];
                rec[R_E] = sm[1];
                rec[R_ST] = sm[2];
                rec[R_SQ] = sm[3];
                rec[R_EQ] = sm[4];
                rec[R_XP] = sm[5];
                rec[R_Y] = sm[6];
                rec[R_ZY] = A(0);
                rec[R_HASY] = A(0);
                if (has_labels && y >= col0 && y < col1) {
                    const int64_t ey = r * V + y;
                    rec[R_ZY] = DFM ? zs_of(A(*df_vy)) : zs_of(Tr::to_acc(xs[ey - wf * EPW]));
                    rec[R_HASY] = A(1);
                }
                if (C > 1) {
                    const uint32_t a0 = smem_addr(myrec);
                    for (int k = 0; k < C; ++k) {
                        const uint32_t ra = map_peer(a0, uint32_t(k));
#pragma unroll
                        for (int i = 0; i < NREC; ++i) st_peer(ra + i * sizeof(A), rec[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NREC; ++i) myrec[i] = rec[i];
                }
            }
            if (C > 1) cluster_barrier();
            if (tid == 0) {
                row_epilogue<A, TEACH, RKL, ENT, CAP, DFM>(p, xch + (xc & 1) * MAX_CLUSTER * NREC, C,
                                                      rank == 0, old_lp, adv, acc, coef, r);
                if (p.tok != nullptr) {  // per-token coefficient on the label column
                    // (the scale is in the coefficients only without softcap;
                    // with softcap it is in the per-element derivative)
                    const A c = A(p.tok[r]) * (CAP ? A(1) : A(p.s));
                    coef[K_PC] -= c;
                    coef[K_BC] -= c;
                }
            }
            ++xc;
            __syncthreads();
        }

        if (!valid && rank == 0 && tid == 0) {  // a masked row's per-token outputs
            if (p.lp_out) p.lp_out[r] = 0.f;
            if (p.rl_out) p.rl_out[r] = 0.f;
        }
        // ---- pass C: the combined gradient, written once (added to grad_out's
        // values when accumulating; a masked row then keeps its values) ----
        if (gg != nullptr && (valid || !p.accumulate)) {
            A lse2 = 0, lseT2 = 0, lsq2 = 0, pc = 0, ps = 0, tc = 0, ts_ = 0, qc = 0, bc = 0;
            if (valid) {
                lse2 = coef[K_LSE2];
                lseT2 = coef[K_LSET2];
                lsq2 = coef[K_LSQ2];
                pc = coef[K_PC];
                ps = coef[K_PS];
                tc = coef[K_TC];
                ts_ = coef[K_TS];
                qc = coef[K_QC];
                bc = coef[K_BC];
            }
            const A dlse = lseT2 - lsq2;
            const int64_t ey = (has_labels && valid && y >= col0 && y < col1) ? r * V + y : -1;
            if (DFM && !p.accumulate) {
                // double-float kernel: fp32 words out.  Non-label elements:
                // pc 2^(zs - lse2) = pc 2^(Z - lse2) 2^d with 2^d (times
                // 2^64) stored by the statistics pass: P = pc 2^(Z - lse2)
                // once per row in double-float, then P (hi + lo) rounded once
                // and scaled by 2^-64 (exactly while normal); the label
                // element in fp64 (it subtracts bc and may cancel).
                // (Accumulating calls take the fp64 kernel; this branch never
                // sees one.)
                DF Pp = {0.f, 0.f};
                int nsc = 0;
                if (valid) {
                    const float vmax = float(coef[DF_VMAX]);
                    DF Zd = df_two_prod(vmax, Kd.h);
                    Zd.l = __fmaf_rn(vmax, Kd.l, Zd.l);
                    const double cz = (double(Zd.h) + double(Zd.l)) - double(lse2);  // <= ~0
                    int nc;
                    const DF Cd = df_exp2(split(cz), nc);
                    const DF Pd = split(double(pc));
                    Pp = df_two_prod(Pd.h, Cd.h);
                    Pp.l = __fmaf_rn(Pd.h, Cd.l, __fmaf_rn(Pd.l, Cd.h, Pp.l));
                    nsc = nc - 64;
                }
                const bool scale_exact = nsc >= -126;
                const float psc = scale_exact ? df_pow2i(nsc) : 0.f;
                for (int w = tid; w < nw; w += nthr) {
                    const int64_t eb = (wf + w) * EPW;
                    const bool full = eb >= e0 && eb + EPW <= e1;
                    float out[4] = {0.f, 0.f, 0.f, 0.f};
                    if (valid) {
                        const float4 k4 = *reinterpret_cast<const float4*>(xs_b + size_t(w) * 16);
                        const uint2 l4 = *reinterpret_cast<const uint2*>(elb + size_t(w) * 4);
                        const float kh[4] = {k4.x, k4.y, k4.z, k4.w};
                        const float kl[4] = {__uint_as_float(l4.x << 16),
                                             __uint_as_float(l4.x & 0xffff0000u),
                                             __uint_as_float(l4.y << 16),
                                             __uint_as_float(l4.y & 0xffff0000u)};
#pragma unroll
                        for (int i = 0; i < EPW; ++i) {
                            DF g = df_two_prod(Pp.h, kh[i]);
                            g.l = __fmaf_rn(Pp.h, kl[i], __fmaf_rn(Pp.l, kh[i], g.l));
                            const float rr = __fadd_rn(g.h, g.l);
                            out[i] = scale_exact ? __fmul_rn(rr, psc) : ldexpf(rr, nsc);
                        }
                        if (ey >= eb && ey < eb + EPW) {
                            const int i = int(ey - eb);
                            const float gy = __double2float_rn(
                                ex2(mul_rn(A(*df_vy), K) - lse2) * pc - bc);
#pragma unroll
                            for (int k = 0; k < EPW; ++k)
                                if (k == i) out[k] = gy;
                        }
                    }
                    if (full) {
                        *reinterpret_cast<float4*>(gg + eb) = make_float4(out[0], out[1], out[2], out[3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < EPW; ++i)
                            if (eb + i >= e0 && eb + i < e1) gg[eb + i] = out[i];
                    }
                }
            } else
            for (int w = tid; w < nw; w += nthr) {
                const int64_t eb = (wf + w) * EPW;
                const bool full = eb >= e0 && eb + EPW <= e1;
                A gv[EPW];
                if (valid) {
                    A v[EPW], u[EPW];
                    Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + size_t(w) * 16), v);
                    if (TEACH)
                        Tr::unpack(*reinterpret_cast<const uint4*>(xs_b + opbytes + size_t(w) * 16),
                                   u);
#pragma unroll
                    for (int i = 0; i < EPW; ++i) {
                        A zs, dz = A(1);
                        if (CAP) {
                            const A th = tnh(v[i] * invc);
                            zs = th * Kc;
                            const A ch = csh(v[i] * invc);  // 1 - tanh^2 = 1 / cosh^2, no cancellation
                            dz = s / (ch * ch);
                        } else {
                            zs = v[i] * K;
                        }
                        const A arg = zs - lse2;
                        A gz = ex2(arg) * (ENT ? pc + ps * arg : pc);
                        if (TEACH) {
                            const A argT = zs * invT - lseT2;
                            const A argq = u[i] * KT - lsq2;
                            A tcoef = tc;
                            if (RKL) {
                                // log2 pT - log2 q from the logit difference,
                                // one rounding at its own scale
                                const A dxu = CAP ? (zs - u[i] * LOG2E) * invT
                                                  : fma(v[i], s, -u[i]) * KT;
                                tcoef = fma(ts_, dxu - dlse, tc);
                            }
                            gz += ex2(argT) * tcoef + qc * ex2(argq);
                        }
                        if (eb + i == ey) gz -= bc;
                        gv[i] = CAP ? gz * dz : gz;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < EPW; ++i) gv[i] = A(0);
                }
                if (full) {
                    if (p.accumulate) {
                        A old[EPW];
                        Tr::unpack(*reinterpret_cast<const uint4*>(gg + eb), old);
#pragma unroll
                        for (int i = 0; i < EPW; ++i) gv[i] = old[i] + gv[i];
                    }
                    *reinterpret_cast<uint4*>(gg + eb) = Tr::pack(gv);
                } else {
#pragma unroll
                    for (int i = 0; i < EPW; ++i)
                        if (eb + i >= e0 && eb + i < e1)
                            gg[eb + i] = Tr::from_acc(p.accumulate ? Tr::to_acc(gg[eb + i]) + gv[i]
                                                                   : gv[i]);
                }
            }
        }
        __syncthreads();  // every thread is done with this stage
        if (tid == 0) issue(it + p.nbuf);
    }

    // A stage whose wait gave up may still receive its copy: wait for it once
    // more (bounded) before the CTA's shared memory goes away.
    if (lost && tid == 0) {
        for (int b = 0; b < p.nbuf; ++b)
            if (lost & (1u << b)) (void)mbar_wait_bounded(smem_addr(&bars[b]), (lost_par >> b) & 1u, p.wait_ns);
    }
    if (rank == 0 && tid == 0) {
        asm volatile("griddepcontrol.launch_dependents;");
        double* out = p.partials + size_t(cid) * NACC;
#pragma unroll
        for (int i = 0; i < NACC; ++i) out[i] = acc[i];
    }
    if (C > 1) cluster_barrier();  // no CTA leaves while a peer may still address it
}

}  // namespace hl
