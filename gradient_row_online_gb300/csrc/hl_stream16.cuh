// hl_stream16.cuh -- the streaming row kernel for bf16 / fp16 logits.
//
// One CTA owns whole rows; no cluster, so no CTA ever waits for another SM.
// A row is streamed through a ring of shared-memory chunk slots twice:
//
//   pass 1  chunks 0 .. K-1: online row statistics.  Each warp keeps one
//           shift per operand for all its lanes (student: s*c*log2e under
//           softcap, else a lazily raised running maximum; teacher: a lazily
//           raised running maximum) and rescales its sums only when a
//           chunk's maximum rises more than TAU above the shift, which after
//           the first chunk almost never happens;
//   merge   with warp-uniform shifts a warp's record is a plain butterfly
//           sum; warp 0 merges the warps' records and derives the row's
//           losses and gradient coefficients (the resident kernel's epilogue);
//   pass 2  chunks K-1 .. 0 (reverse order, so the chunks read most recently
//           -- the ones most likely still in L2 -- come back first): the
//           combined gradient, written once from registers.
//
// Full chunks in the narrow softcap tier (or without softcap) take a hot
// path: four words per thread, unrolled, no per-word predicate, no tier
// dispatch.  Partial chunks and the wider tiers take a rolled cold path.  The
// label column's logit is read once per row from global memory, and its
// gradient element is patched after the row's last chunk by the thread that
// wrote its word.
//
// Softcap transform, per (warp, chunk): zs = s*c*log2e*tanh(x/c) is x * Q(x^2)
// with the scale folded into the polynomial Q when the chunk's max |x| / c is
// within a fitted range (tier A: degree 3 on |y| <= 0.45; tier B: degree 5
// on |y| <= 0.8), else tanh comes from ex2 + rcp (tier X).  Pass 1 records
// each warp's tier per chunk; pass 2, which visits the same elements with the
// same threads, reuses it.
//
// The chunk stream (row, pass, chunk) is one sequence per CTA; the ring slot
// and phase of each entry advance incrementally, and a thread of the last
// warp to finish an entry issues the bulk copy of the entry S places later
// into the same slot, so copies for the next row start while this row
// finishes.  The second read of a row is served by L2 when the row's chunks
// are still resident; the DRAM bytes it costs are measured, not assumed.
//
// Rows must be 16-byte aligned (V * 2 a multiple of 16); the planner sends
// other shapes to the resident kernel, which handles ragged rows.
#pragma once
#include "hl_rows16.cuh"

namespace hl {

template <int I>
struct IntC {
    static constexpr int value = I;
};

// Maximum of v over the warp, in every lane (order-preserving integer key).
__device__ __forceinline__ float warp_max_f(float v) {
    int k = __float_as_int(v);
    k = k >= 0 ? k : k ^ 0x7fffffff;
    k = __reduce_max_sync(0xffffffffu, k);
    return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

// Largest rise (base-2 units) of a value above its running shift before the
// sums are rescaled: terms stay below 2^TAU, far from fp32 overflow.
constexpr float STREAM_TAU = 16.f;

// A gradient word stored with the streaming (evict-first) cache hint: its
// lines are written once and never read here, so they should not push the
// rows' first-pass lines out of L2 (taken on teacher rows: measured, all-in
// 11.70-11.75 -> 11.68 ms; distillation, with its hinted copies, 2.67 ->
// 2.64 ms).
__device__ __forceinline__ void st_stream(void* ptr, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

template <typename DT, int FEAT, bool ACC>
__global__ void __launch_bounds__(THREADS, 1) stream_kernel16(const __grid_constant__ Params p) {
    using P16 = Pack16<DT>;
    constexpr int EPW = 8;
    constexpr int ES = 2;
    constexpr bool TEACH = (FEAT & F_TEACH) != 0;
    constexpr bool RKL = (FEAT & F_RKL) != 0;
    constexpr bool ENT = (FEAT & F_ENT) != 0;
    constexpr bool CAP = (FEAT & F_SOFTCAP) != 0;
    constexpr bool DCE = TEACH && (FEAT & F_DCE) != 0;
    constexpr bool ENTG = ENT && (FEAT & F_ENTG) != 0;
    // T = 2 exactly (no softcap, no entropy): 2^d = (2^(d/2))^2, so the
    // probabilities at T = 1 and at T come from one exponential
    constexpr bool T2 = TEACH && !CAP && !ENT && (FEAT & F_T2) != 0;
    constexpr int OPS = TEACH ? 2 : 1;

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = int(blockDim.x), nwarps = nthr >> 5;
    const int S = p.nbuf;                 // chunk slots in the ring
    const int CH = int(p.L);              // elements per chunk (a multiple of 8 * nthr)
    const uint32_t opbytes = uint32_t(CH) * ES;
    const uint32_t slot_bytes = opbytes * OPS;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(slot_bytes) * S);
    float* acc = reinterpret_cast<float*>(bars + MAX_STAGES);  // [2][NACC]: sums, compensations
    float* xch = acc + 2 * NACC;                                // per-warp records of a row
    float* red = xch + 2 * MAX_CLUSTER * NREC;
    float* redmax = red + NWARPS * NREC;
    float* coefs = redmax + 2 * NWARPS;
    RowLoss* rls = reinterpret_cast<RowLoss*>(coefs + 16);  // a row's losses, summed after the merge
    int* done = reinterpret_cast<int*>(coefs + 32);     // [MAX_STAGES] warps finished per slot
    static_assert(sizeof(RowCoef) <= 16 * sizeof(float) && sizeof(RowLoss) <= 16 * sizeof(float),
                  "coefficient / row-loss areas");

    const int64_t N = p.N, V = p.V;
    const int K = int((V + CH - 1) / CH);                // chunks per row
    const int K2x = 2 * K;                               // stream entries per row
    const int64_t G = gridDim.x;
    const DT* __restrict__ xg = static_cast<const DT*>(p.x);
    const DT* __restrict__ tg = static_cast<const DT*>(p.t);
    DT* gg = static_cast<DT*>(p.g);

    const float LOG2E = 1.4426950408889634f;
    const float s = p.s;
    const float K1 = s * LOG2E;
    const float invc = CAP ? 1.f / p.softcap : 0.f;
    const float A2 = CAP ? 2.f * LOG2E * invc : 0.f;
    const float Kc = CAP ? s * p.softcap * LOG2E : 0.f;
    const float invT = 1.f / p.T;
    const float KT = LOG2E * invT;
    // softcap: the student shift is the constant Kc when every shifted term,
    // at temperature 1 and T, stays above 2^-120 (|zs| <= Kc); otherwise it
    // follows the running maximum like the teacher's
    const bool fixed_shift = CAP && Kc * fmaxf(1.f, invT) <= 60.f;
    // tier bounds on max |x| (tanh argument x / c); the narrow tier's fit
    // error (2.4e-7 relative) stays below fp32 rounding of exp(zs) only while
    // |zs| is moderate, so it is used for Kc <= 48 alone
    const float XA = (CAP && Kc <= 48.f) ? HL_TANH_A_Y0 * p.softcap : 0.f;
    const float XB = CAP ? HL_TANH_B_Y0 * p.softcap : 0.f;
    // zs = x * Q(x^2): Q_k = s * log2e * C_k / c^(2k), formed in double
    f2 QA[4], QB[6];  // QB: staged in shared memory below (rarely needed)
    {
        const double ic2 = CAP ? 1.0 / (double(p.softcap) * double(p.softcap)) : 0.0;
        const double ca[4] = {HL_TANH_A_C0, HL_TANH_A_C1, HL_TANH_A_C2, HL_TANH_A_C3};
        const double cb[6] = {HL_TANH_B_C0, HL_TANH_B_C1, HL_TANH_B_C2,
                              HL_TANH_B_C3, HL_TANH_B_C4, HL_TANH_B_C5};
        double f = double(s) * 1.4426950408889634;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
            if (k < 4) QA[k] = pk1(float(ca[k] * f));
            QB[k] = pk1(float(cb[k] * f));
            f *= ic2;
        }
    }
    const f2 K2 = pk1(K1), A22 = pk1(A2), Kc2 = pk1(Kc), invT2 = pk1(invT), KT2 = pk1(KT);
    const f2 K2h = pk1(T2 ? 0.5f * K1 : 0.f);  // T = 2: the first pass forms d / 2 directly
    const f2 KinvT2 = pk1(K1 * invT);
    const f2 m2 = pk1(CAP ? -1.f / (Kc * Kc) : 0.f), one2 = pk1(1.f);
    const f2 z2 = pk1(0.f);

    auto zs1 = [&](float v) -> float {
        return CAP ? __fmul_rn(tanh_a2x_1(__fmul_rn(v, A2)), Kc) : __fmul_rn(v, K1);
    };
    // zs + nshift of a pair (pass 1), by tier
    // the wide-tier and exp-tier constants live in shared memory (the `red`
    // area, unused here) and are read at each use (volatile: never hoisted into
    // registers), so the common tier keeps all registers for itself
    f2* rare = reinterpret_cast<f2*>(red);  // QB[0..5], A22, Kc2
    const volatile f2* cst = rare;
    auto shifted = [&](f2 xv, f2 nshift, auto tierc) -> f2 {
        constexpr int TI = CAP ? decltype(tierc)::value : -1;
        if constexpr (TI < 0) {
            return fma2(xv, K2, nshift);
        } else if constexpr (TI == 0) {
            const f2 u = mul2(xv, xv);
            f2 q = fma2(u, QA[3], QA[2]);
            q = fma2(q, u, QA[1]);
            q = fma2(q, u, QA[0]);
            return fma2(xv, q, nshift);
        } else if constexpr (TI == 1) {
            const f2 u = mul2(xv, xv);
            f2 q = fma2(u, cst[5], cst[4]);
            q = fma2(q, u, cst[3]);
            q = fma2(q, u, cst[2]);
            q = fma2(q, u, cst[1]);
            q = fma2(q, u, cst[0]);
            return fma2(xv, q, nshift);
        } else {
            return fma2(tanh_from_ex2_arg(mul2(xv, cst[6])).th, cst[7], nshift);
        }
    };
    // zs and 1 - tanh^2 of a pair (pass 2, softcap), by tier
    auto zs_omt = [&](f2 xv, f2& zs, f2& omt, auto tierc) {
        constexpr int TI = decltype(tierc)::value;
        if constexpr (TI == 0 || TI == 1) {
            const f2 u = mul2(xv, xv);
            f2 q;
            if constexpr (TI == 0) {
                q = fma2(u, QA[3], QA[2]);
                q = fma2(q, u, QA[1]);
                q = fma2(q, u, QA[0]);
            } else {
                q = fma2(u, cst[5], cst[4]);
                q = fma2(q, u, cst[3]);
                q = fma2(q, u, cst[2]);
                q = fma2(q, u, cst[1]);
                q = fma2(q, u, cst[0]);
            }
            zs = mul2(xv, q);
            omt = fma2(zs, mul2(zs, m2), one2);  // 1 - (zs / Kc)^2; |tanh| <= 0.67 here
        } else {
            const TanhD2 td = tanh_from_ex2_arg(mul2(xv, cst[6]));
            zs = mul2(td.th, cst[7]);
            omt = td.omt;
        }
    };

    // stream position -> copy: entry jl of row r (jl < K: pass-1 chunk jl;
    // else pass-2 chunk 2K-1-jl) into ring slot sl
    auto issue = [&](int sl, int64_t r, int jl) {
        if (r >= N) return;
        const int c = jl < K ? jl : K2x - 1 - jl;
        const uint32_t bar = smem_addr(&bars[sl]);
        const int64_t c0 = int64_t(c) * CH;
        const int64_t len = (V - c0) < CH ? (V - c0) : CH;
        const uint32_t bytes = uint32_t(len * ES);
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, bytes * OPS);
#ifdef HL_FAULT_INJECT
        if (r == p.drop_row && jl == 0) return;  // pass-1 chunk 0 never comes
#endif
        const uint32_t dst = smem_addr(smem + size_t(sl) * slot_bytes);
        if constexpr ((FEAT & F_L2P) != 0) {
            // the teacher's first-pass copies stay in L2 for the second
            // pass's re-read; second-pass copies (their last use) go first
            // (the student's first pass as well was measured slower)
            uint64_t pol;
            if (jl < K) {
                asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
                bulk_g2s(dst, xg + r * V + c0, bytes, bar);
            } else {
                asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
                bulk_g2s_hint(dst, xg + r * V + c0, bytes, bar, pol);
            }
            if (TEACH) bulk_g2s_hint(dst + opbytes, tg + r * V + c0, bytes, bar, pol);
        } else {
            bulk_g2s(dst, xg + r * V + c0, bytes, bar);
            if (TEACH) bulk_g2s(dst + opbytes, tg + r * V + c0, bytes, bar);
        }
    };
    // the entry `ahead` places after (r, jl)
    auto advance = [&](int64_t& r, int& jl, int ahead) {
        jl += ahead;
        while (jl >= K2x) {
            jl -= K2x;
            r += G;
        }
    };

    if (tid == 0) {
        for (int b = 0; b < S; ++b) {
            mbar_init(smem_addr(&bars[b]), 1);
            done[b] = 0;
        }
        fence_mbar_init();
        for (int i = 0; i < 2 * NACC; ++i) acc[i] = 0.f;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the count kernel has completed
        coefs[KK_SLOT] = *p.kscale;
#pragma unroll
        for (int i = 0; i < 6; ++i) rare[i] = QB[i];
        rare[6] = A22;
        rare[7] = Kc2;
    }
    __syncthreads();
    if (tid == 0) {
        for (int j = 0; j < S; ++j) {
            int64_t r = blockIdx.x;
            int jl = 0;
            advance(r, jl, j);
            issue(j, r, jl);
        }
    }

    int slot = 0;
    uint32_t phase = 0;               // ring slot and phase parity of the next entry
    uint32_t lost = 0, lost_par = 0;  // slots (and phase parities) whose wait gave up
    // wait for the current entry's slot; returns its shared-memory base
    auto acquire = [&]() -> const unsigned char* {
        if (!mbar_wait_bounded(smem_addr(&bars[slot]), phase, p.wait_ns)) {
            lost |= 1u << slot;
            lost_par = (lost_par & ~(1u << slot)) | (phase << slot);
            if (lane == 0) atomicOr(p.err, E_TIMEOUT);
        }
        return smem + size_t(slot) * slot_bytes;
    };
    // this warp is done with the current entry (row r, position jl); the last
    // warp refills the slot with the entry S places later; then step the ring
    auto release = [&](int64_t r, int jl) {
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const int old = atomicAdd(&done[slot], 1);
            if (old + 1 == nwarps) {
                // every warp has left this slot; the next use can count again
                // (the copy below completes before any warp touches the slot)
                done[slot] = 0;
                __threadfence_block();
                advance(r, jl, S);
                issue(slot, r, jl);
            }
        }
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    };

    const bool has_labels = p.labels != nullptr;
    const bool need_side = (p.flags & (L_GRPO | L_GRPO_STATS)) != 0;
    const int WPT = CH / (EPW * nthr);  // words per thread per chunk (full chunks)

    // A row's side inputs (label, old log-prob, advantage) are staged a row
    // ahead, per warp, in shared memory after the rare constants: lane 0
    // loads the next row's during the merge and stores them after it, so a
    // row starts on a shared-memory read instead of a global load.
    struct Side {
        int64_t y;
        float o, a;
    };
    static_assert(16 + (2 + 2) * NWARPS <= NWARPS * NREC, "side-input stash");
    int64_t* ystash = reinterpret_cast<int64_t*>(red + 16);     // [NWARPS]
    float* sstash = reinterpret_cast<float*>(ystash + NWARPS);  // [NWARPS][2]
    auto side_load = [&](int64_t rn) -> Side {
        Side sd{0, 0.f, 0.f};
        if (rn < N) {
            if (has_labels) sd.y = p.labels[rn];
            if (need_side) {
                sd.o = p.old_lp[rn];
                sd.a = p.adv[rn];
            }
        }
        return sd;
    };
    auto side_store = [&](const Side& sd) {
        ystash[warp] = sd.y;
        sstash[2 * warp] = sd.o;
        sstash[2 * warp + 1] = sd.a;
    };
    if (lane == 0) side_store(side_load(blockIdx.x));

    for (int64_t r = blockIdx.x; r < N; r += G) {
        __syncwarp();
        const int64_t y = ystash[warp];
        const float old_lp = sstash[2 * warp];
        const float adv = sstash[2 * warp + 1];
        __syncwarp();
        const bool valid = !has_labels || (y >= 0 && y < V);
        if (has_labels && y >= V && tid == 0) atomicOr(p.err, E_LABEL);

        if (!valid) {  // a masked row: consume its entries, write exact +0
            if (tid == 0) write_row_zero(p, r);
            Side nxt{};
            if (lane == 0) nxt = side_load(r + G);
            for (int jl = 0; jl < K2x; ++jl) {
                acquire();
                const int cc = jl < K ? jl : K2x - 1 - jl;
                if (jl >= K && gg != nullptr && !ACC) {  // kept when accumulating
                    const int64_t c0 = int64_t(cc) * CH;
                    const int nwc = int(((V - c0) < CH ? (V - c0) : CH) / EPW);
                    for (int w = tid; w < nwc; w += nthr)
                        *reinterpret_cast<uint4*>(gg + r * V + c0 + int64_t(w) * EPW) =
                            make_uint4(0, 0, 0, 0);
                }
                release(r, jl);
            }
            if (lane == 0) side_store(nxt);
            continue;
        }

        // the label column: thread 0 reads its logit now and uses it at the
        // merge (so the read is not waited for); the thread whose pass-2 word
        // holds it patches that element after the row's last chunk
        const int yc = has_labels ? int(y / CH) : -1;
        const int yin = has_labels ? int(y - int64_t(yc) * CH) : 0;
        const int ywd = yin / EPW;
        const bool yown = has_labels && ywd >= tid && (ywd - tid) % nthr == 0 &&
                          (ywd - tid) / nthr < WPT;
        uint16_t xy_bits = 0;
        if (has_labels && tid == 0) xy_bits = reinterpret_cast<const uint16_t*>(xg)[r * V + y];

        // ---------------- pass 1: online statistics ----------------
        float zm = fixed_shift ? Kc : -CUDART_INF_F, um = -CUDART_INF_F;
        f2 S2 = z2, E2 = z2, ST2 = z2, Sq2 = z2, Eq2 = z2, Xp2 = z2, Y2 = z2;
        uint64_t tiers = 0;  // softcap: 2 bits per chunk (chunks 0..31) of this warp
        int tier_hi = 0;     // softcap: highest tier of chunks 32.. of this warp
        const bool need_sx = !CAP || !fixed_shift;
        // one pair's contribution to the sums, given its shifted logit d
        auto accum = [&](f2 d, uint32_t tbits, f2 num2) {
            f2 e, dT, eT;
            if constexpr (T2) {
                dT = d;  // the caller passes d / 2
                eT = ex2p(dT);
                e = mul2(eT, eT);
            } else {
                e = ex2p(d);
            }
            S2 = add2(S2, e);
            if (ENT) E2 = fma2(e, d, E2);
            if (TEACH) {
                if constexpr (!T2) {
                    dT = mul2(d, invT2);
                    eT = ex2p(dT);
                }
                ST2 = add2(ST2, eT);
                const f2 du = fma2(P16::unpack(tbits), KT2, num2);
                const f2 eq = ex2p(du);
                Sq2 = add2(Sq2, eq);
                if (DCE) Eq2 = fma2(eq, du, Eq2);
                const f2 wd = sub2(du, dT);
                Xp2 = fma2(eq, wd, Xp2);
                if (RKL) Y2 = fma2(eT, wd, Y2);
            }
        };
        for (int c = 0; c < K; ++c) {
            const unsigned char* sb = acquire();
            const int64_t c0 = int64_t(c) * CH;
            const int nwc = int(((V - c0) < CH ? (V - c0) : CH) / EPW);
            // a full chunk gives every thread four words: the hot path
            const bool full = WPT == 4 && nwc == 4 * nthr;
            const bool mine = full || tid < nwc;
            // chunk maxima of this thread's words on packed pairs: max |x|
            // (softcap tier), signed max x (shift, unless fixed), max t
            uint32_t ma = 0u, ms = P16::NEG_INF2, mt = P16::NEG_INF2;
            auto maxw = [&](const uint4& a, const uint4& b, auto sxc) {
                if (CAP)
                    ma = P16::absmax2(ma, P16::absmax2(P16::absmax2(a.x, a.y),
                                                       P16::absmax2(a.z, a.w)));
                if (decltype(sxc)::value)
                    ms = P16::max2(ms, P16::max2(P16::max2(a.x, a.y), P16::max2(a.z, a.w)));
                if (TEACH)
                    mt = P16::max2(mt, P16::max2(P16::max2(b.x, b.y), P16::max2(b.z, b.w)));
            };
            uint4 xw[4], tw[4];
            if (full) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int w = tid + i * nthr;
                    xw[i] = *reinterpret_cast<const uint4*>(sb + size_t(w) * 16);
                    if (TEACH) tw[i] = *reinterpret_cast<const uint4*>(sb + opbytes + size_t(w) * 16);
                    else tw[i] = make_uint4(0, 0, 0, 0);
                }
                if (need_sx) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) maxw(xw[i], tw[i], BoolC<true>{});
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) maxw(xw[i], tw[i], BoolC<false>{});
                }
            } else {
#pragma unroll 1
                for (int i = 0; i < WPT; ++i) {
                    const int w = tid + i * nthr;
                    if (w >= nwc) break;
                    const uint4 a = *reinterpret_cast<const uint4*>(sb + size_t(w) * 16);
                    const uint4 b = TEACH ? *reinterpret_cast<const uint4*>(sb + opbytes + size_t(w) * 16)
                                          : make_uint4(0, 0, 0, 0);
                    maxw(a, b, BoolC<true>{});
                }
            }
            float ca, cb;
            // lazy, warp-uniform shifts: raise a shift only when the warp's
            // chunk maximum exceeds it by TAU
            float nz = zm, nu = um;
            bool mv = false;
            if (need_sx) {
                upk(P16::unpack(ms), ca, cb);
                const float wmx = warp_max_f(mine ? fmaxf(ca, cb) : -CUDART_INF_F);
                if (wmx > -CUDART_INF_F) {
                    const float bz = zs1(wmx);
                    if (bz > zm + STREAM_TAU) {
                        nz = bz;
                        mv = true;
                    }
                }
            }
            if (TEACH) {
                upk(P16::unpack(mt), ca, cb);
                const float wmt = warp_max_f(mine ? fmaxf(ca, cb) : -CUDART_INF_F);
                if (wmt > -CUDART_INF_F) {
                    const float bu = __fmul_rn(wmt, KT);
                    if (bu > um + STREAM_TAU) {
                        nu = bu;
                        mv = true;
                    }
                }
            }
            if (mv) {  // warp-uniform
                const float d = (zm == -CUDART_INF_F) ? 0.f : zm - nz;
                const float du = (um == -CUDART_INF_F) ? 0.f : um - nu;
                const float al = exp2f(d), dTv = d * invT;
                const f2 al2 = pk1(al), d2 = pk1(d);
                if (ENT) E2 = mul2(al2, fma2(d2, S2, E2));
                S2 = mul2(al2, S2);
                if (TEACH) {
                    const float alT = exp2f(dTv), be = exp2f(du);
                    const f2 alT2 = pk1(alT), be2 = pk1(be), du2 = pk1(du);
                    const f2 w2 = pk1(du - dTv);
                    Xp2 = mul2(be2, fma2(w2, Sq2, Xp2));
                    if (DCE) Eq2 = mul2(be2, fma2(du2, Sq2, Eq2));
                    if (RKL) Y2 = mul2(alT2, fma2(w2, ST2, Y2));
                    ST2 = mul2(alT2, ST2);
                    Sq2 = mul2(be2, Sq2);
                }
                zm = nz;
                um = nu;
            }
            // softcap tier of this warp's words in the chunk
            int tier = 0;
            if (CAP) {
                upk(P16::unpack(ma), ca, cb);
                const float cx = fmaxf(fabsf(ca), fabsf(cb));
                tier = __all_sync(0xffffffffu, cx <= XA) ? 0
                       : __all_sync(0xffffffffu, cx <= XB) ? 1 : 2;
                if (c < 32) tiers |= uint64_t(tier) << (2 * c);
                else tier_hi = tier > tier_hi ? tier : tier_hi;
            }
            const f2 nzm2 = pk1(-zm), num2 = pk1(-um);
            const f2 nzmh2 = pk1(T2 ? -0.5f * zm : 0.f);
            if (full && tier == 0) {
                // hot path: four words, the narrow tier (or no softcap), unrolled
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t xa[4] = {xw[i].x, xw[i].y, xw[i].z, xw[i].w};
                    const uint32_t tb[4] = {tw[i].x, tw[i].y, tw[i].z, tw[i].w};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        if constexpr (T2)
                            accum(fma2(P16::unpack(xa[kk]), K2h, nzmh2), tb[kk], num2);
                        else
                            accum(shifted(P16::unpack(xa[kk]), nzm2, IntC<0>{}), tb[kk], num2);
                }
            } else {
                // cold path: a partial chunk or a wider tier, one word at a time
#pragma unroll 1
                for (int i = 0; i < WPT; ++i) {
                    const int w = tid + i * nthr;
                    if (w >= nwc) break;
                    const uint4 a = *reinterpret_cast<const uint4*>(sb + size_t(w) * 16);
                    const uint4 b = TEACH ? *reinterpret_cast<const uint4*>(sb + opbytes + size_t(w) * 16)
                                          : make_uint4(0, 0, 0, 0);
                    const uint32_t xa[4] = {a.x, a.y, a.z, a.w};
                    const uint32_t tb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const f2 xv = P16::unpack(xa[kk]);
                        f2 d;
                        if (T2) d = fma2(xv, K2h, nzmh2);
                        else if (!CAP || tier == 0) d = shifted(xv, nzm2, IntC<0>{});
                        else if (tier == 1) d = shifted(xv, nzm2, IntC<1>{});
                        else d = shifted(xv, nzm2, IntC<2>{});
                        accum(d, tb[kk], num2);
                    }
                }
            }
            release(r, c);
        }
        const float zy = (has_labels && tid == 0) ? zs1(P16::to_f(xy_bits)) : 0.f;
        const float hasy = (has_labels && tid == 0) ? 1.f : 0.f;

        // ---------------- merge: threads -> warps -> row ----------------
        Side nxt{};
        if (lane == 0) nxt = side_load(r + G);  // stored after the merge
        // the shifts are warp-uniform, so a warp's record is a plain sum
        float v[9] = {hsum(S2), hsum(E2), hsum(ST2), hsum(Sq2), hsum(Eq2), hsum(Xp2),
                      -hsum(Y2), zy, hasy};
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int i = 0; i < 9; ++i) {
                if (i == 1 && !ENT) continue;
                if ((i >= 2 && i <= 5) && !TEACH) continue;
                if (i == 4 && !DCE) continue;
                if (i == 6 && !RKL) continue;
                v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
            }
        if (lane == 0) {
            float* rec = xch + warp * NREC;
            rec[R_ZM] = zm;
            rec[R_UM] = um;
            rec[R_S] = v[0];
            rec[R_E] = ENT ? v[1] : 0.f;
            rec[R_ST] = TEACH ? v[2] : 0.f;
            rec[R_SQ] = TEACH ? v[3] : 0.f;
            rec[R_EQ] = DCE ? v[4] : 0.f;
            rec[R_XP] = TEACH ? v[5] : 0.f;
            rec[R_Y] = RKL ? v[6] : 0.f;
            rec[R_ZY] = v[7];
            rec[R_HASY] = v[8];
        }
        __syncthreads();
        // the row's losses wait in shared memory and are added once the
        // coefficients are out
        if (warp == 0) {
            const RowCoef kw = row_epilogue16<TEACH, RKL, ENT, CAP, true>(
                p, xch, nwarps, false, old_lp, adv, acc, lane, r, coefs[KK_SLOT], rls);
            if (lane == 0) *reinterpret_cast<RowCoef*>(coefs) = kw;
        }
        __syncthreads();
        if (lane == 0) side_store(nxt);
        if (tid == 0) row_accumulate(p, *rls, acc, r);
        const RowCoef k = *reinterpret_cast<const RowCoef*>(coefs);

        // ---------------- pass 2: the gradient, reverse chunk order ----------------
        // exponentials offset by 2^sg, coefficients scaled by 2^-sg
        const ShiftCoef h = shift_coefs(k, ENTG);
        const float dlse = k.lseT2 - k.lsq2;
        const f2 nlse2 = pk1(h.nlse), nlseT2 = pk1(h.nlseT), nlsq2 = pk1(h.nlsq);
        const f2 pc2 = pk1(h.pc), ps2 = pk1(h.ps), tc2 = pk1(h.tc), ts2 = pk1(h.ts);
        const f2 qc2 = pk1(h.qc), s2 = pk1(s), ndlse2 = pk1(-dlse);
        const f2 nKT2 = pk1(-KT);
        // T = 2: hh = 2^((x K1 + nlse) / 2), so p 2^sg = hh^2 and pT 2^sg = hh cT
        // with cT = 2^(nlseT - nlse / 2) (a row constant, from the library
        // exp2); the gradient is hh (hh pc + cT tco) + q qc, and with reverse
        // KL cT tco = cT (ts (dxu - dlse) + tc), dxu = (x s - t) KT, is
        // x A + (t B + C)
        const float cT = T2 ? exp2f(h.nlseT - 0.5f * h.nlse) : 0.f;
        const f2 Kh2 = pk1(T2 ? 0.5f * K1 : 0.f), nlseh2 = pk1(T2 ? 0.5f * h.nlse : 0.f);
        const f2 rA2 = pk1(T2 && RKL ? cT * h.ts * s * KT : 0.f);
        const f2 rB2 = pk1(T2 && RKL ? -cT * h.ts * KT : 0.f);
        const f2 rC2 = pk1(T2 ? cT * (RKL ? fmaf(-h.ts, dlse, h.tc) : h.tc) : 0.f);
        // accumulating: the label element's existing value, read before this
        // row's word stores overwrite it
        float old_y = 0.f;
        if (ACC && yown && gg != nullptr)
            old_y = P16::to_f(reinterpret_cast<const uint16_t*>(gg)[r * V + y]);
        // the gradient of one word (8 elements), without the label term
        auto grad_word = [&](uint4 a, uint4 b, uint4 ow, auto tierc) -> uint4 {
            const uint32_t xa[4] = {a.x, a.y, a.z, a.w};
            const uint32_t tb[4] = {b.x, b.y, b.z, b.w};
            const uint32_t oa[4] = {ow.x, ow.y, ow.z, ow.w};
            uint32_t out[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const f2 xv = P16::unpack(xa[kk]);
                f2 omt = z2, g;
                if constexpr (T2) {
                    const f2 tv = P16::unpack(tb[kk]);
                    const f2 hh = ex2p(fma2(xv, Kh2, nlseh2));
                    const f2 q = ex2p(fma2(tv, KT2, nlsq2));
                    f2 tcoT = rC2;
                    if constexpr (RKL) tcoT = fma2(xv, rA2, fma2(tv, rB2, rC2));
                    g = fma2(hh, fma2(hh, pc2, tcoT), mul2(q, qc2));
                } else {
                    f2 zs = z2, arg, argT = z2;
                    if constexpr (CAP) {
                        zs_omt(xv, zs, omt, tierc);
                        arg = add2(zs, nlse2);
                        if (TEACH) argT = fma2(zs, invT2, nlseT2);
                    } else {
                        arg = fma2(xv, K2, nlse2);
                        if (TEACH) argT = fma2(xv, KinvT2, nlseT2);
                    }
                    g = mul2(ex2p(arg), ENTG ? fma2(ps2, arg, pc2) : pc2);
                    if (TEACH) {
                        const f2 tv = P16::unpack(tb[kk]);
                        const f2 pT = ex2p(argT);
                        const f2 q = ex2p(fma2(tv, KT2, nlsq2));
                        f2 tco = tc2;
                        if (RKL) {
                            // log pT - log q from the logit difference
                            const f2 dxu = CAP ? fma2(zs, invT2, mul2(tv, nKT2))
                                               : mul2(fma2(xv, s2, sub2(z2, tv)), KT2);
                            tco = fma2(ts2, add2(dxu, ndlse2), tc2);
                        }
                        g = fma2(pT, tco, g);
                        g = fma2(q, qc2, g);
                    }
                }
                // dz/dx = s (1 - tanh^2); s is already in the coefficients
                const f2 gw = CAP ? mul2(g, omt) : g;
                out[kk] = P16::pack(ACC ? add2(P16::unpack(oa[kk]), gw) : gw);
            }
            return make_uint4(out[0], out[1], out[2], out[3]);
        };
        for (int cr = 0; cr < K; ++cr) {
            const int c = K - 1 - cr;
            const unsigned char* sb = acquire();
            if (gg != nullptr) {
                const int64_t c0 = int64_t(c) * CH;
                const int nwc = int(((V - c0) < CH ? (V - c0) : CH) / EPW);
                const bool full = WPT == 4 && nwc == 4 * nthr;
                DT* grow = gg + r * V + c0;
                const int tier = !CAP ? 0 : c < 32 ? int((tiers >> (2 * c)) & 3u) : tier_hi;
                if (full && tier == 0) {
                    // hot path: four words, the narrow tier (or no softcap), unrolled
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int w = tid + i * nthr;
                        uint4 ow = make_uint4(0, 0, 0, 0);
                        if (ACC) ow = *reinterpret_cast<const uint4*>(grow + int64_t(w) * EPW);
                        const uint4 a = *reinterpret_cast<const uint4*>(sb + size_t(w) * 16);
                        const uint4 b = TEACH ? *reinterpret_cast<const uint4*>(sb + opbytes + size_t(w) * 16)
                                              : make_uint4(0, 0, 0, 0);
                        if constexpr (TEACH)
                            st_stream(grow + int64_t(w) * EPW, grad_word(a, b, ow, IntC<0>{}));
                        else
                            *reinterpret_cast<uint4*>(grow + int64_t(w) * EPW) =
                                grad_word(a, b, ow, IntC<0>{});
                    }
                } else {
                    // cold path: a partial chunk or a wider tier, one word at a time
#pragma unroll 1
                    for (int i = 0; i < WPT; ++i) {
                        const int w = tid + i * nthr;
                        if (w >= nwc) break;
                        uint4 ow = make_uint4(0, 0, 0, 0);
                        if (ACC) ow = *reinterpret_cast<const uint4*>(grow + int64_t(w) * EPW);
                        const uint4 a = *reinterpret_cast<const uint4*>(sb + size_t(w) * 16);
                        const uint4 b = TEACH ? *reinterpret_cast<const uint4*>(sb + opbytes + size_t(w) * 16)
                                              : make_uint4(0, 0, 0, 0);
                        uint4 o;
                        if (!CAP || tier == 0) o = grad_word(a, b, ow, IntC<0>{});
                        else if (tier == 1) o = grad_word(a, b, ow, IntC<1>{});
                        else o = grad_word(a, b, ow, IntC<2>{});
                        if constexpr (TEACH) st_stream(grow + int64_t(w) * EPW, o);
                        else *reinterpret_cast<uint4*>(grow + int64_t(w) * EPW) = o;
                    }
                }
            }
            release(r, K2x - 1 - c);
        }
        // the label column: the thread whose word held it recomputes that one
        // element with the label term (inputs re-read from global memory) and
        // overwrites it; program order puts this store after its word store
        if (yown && gg != nullptr) {
            // the coefficients again from shared memory (no register carries them
            // through the chunk loop; they stay until the next row's merge)
            const RowCoef k = *reinterpret_cast<const RowCoef*>(coefs);
            const ShiftCoef h = shift_coefs(k, ENTG);
            const float dlse = k.lseT2 - k.lsq2;
            const float xv1 = P16::to_f(reinterpret_cast<const uint16_t*>(xg)[r * V + y]);
            float zs, om1 = 1.f;
            if (CAP) zs = __fmul_rn(tanh_a2x_1(__fmul_rn(xv1, A2), &om1), Kc);
            else zs = __fmul_rn(xv1, K1);
            const float arg = zs + h.nlse;
            float g1 = ex2f(arg) * (ENTG ? fmaf(h.ps, arg, h.pc) : h.pc);
            if (TEACH) {
                const float tv1 = P16::to_f(reinterpret_cast<const uint16_t*>(tg)[r * V + y]);
                const float pT = ex2f(fmaf(zs, invT, h.nlseT));
                const float q = ex2f(fmaf(tv1, KT, h.nlsq));
                float tco = h.tc;
                if (RKL) {
                    const float dxu = CAP ? fmaf(tv1, -LOG2E, zs) * invT : fmaf(xv1, s, -tv1) * KT;
                    tco = fmaf(h.ts, dxu - dlse, h.tc);
                }
                g1 = fmaf(pT, tco, g1);
                g1 = fmaf(q, h.qc, g1);
            }
            g1 -= k.bc;
            if (CAP) g1 *= om1;
            if (ACC) g1 = old_y + g1;
            reinterpret_cast<uint16_t*>(gg)[r * V + y] = P16::from_f(g1);
        }
    }

    // a slot whose wait gave up may still receive its copy: wait once more
    // (bounded) before the CTA's shared memory goes away
    if (lost && tid == 0) {
        for (int b = 0; b < S; ++b)
            if (lost & (1u << b)) (void)mbar_wait_bounded(smem_addr(&bars[b]), (lost_par >> b) & 1u, p.wait_ns);
    }
    if (tid == 0) {
        store_partials(acc, p.partials + size_t(blockIdx.x) * NACC);
        asm volatile("griddepcontrol.launch_dependents;");  // the finalize kernel may launch
    }
}

}  // namespace hl
