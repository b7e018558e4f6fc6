// hl_onepass.cu -- the loss's gradient pass alone, for logits whose first-pass
// statistics came out of the LM-head GEMM's epilogue
// (headloss_lmhead_logits_rowstats): headloss_forward_backward_rowstats.
//
// The fused LM head of the pages (ServiceNow Fast-LLM PR #549,
// "Correctness": the LM head and tied embeddings) computes the logits and the
// loss back to back.  On GB300 the GEMM's epilogue holds each output tile in
// TMEM, one row per thread, so it can also emit the tile's contribution to
// the row's softmax statistics; the loss then needs a single read of the
// logits and a single write of the gradient: no statistics pass, no second
// read.  The statistics it consumes are, per (row, 256-column tile), the base-2
// record (m2, S, E, X) of zs = s c tanh(x / c) log2(e) (c = 0: s x log2(e)):
// m2 = max zs, S = sum 2^(zs - m2), E = sum 2^(zs - m2) (zs - m2), X = max |x|.
// These cover the label-based losses (CE, z-loss, GRPO and its statistics,
// entropy).  With a teacher (from-distribution CE, forward KL) two more come
// in: the student tile's S_T = sum 2^((zs - m2) / T) and the teacher GEMM's
// record of ut = t log2(e) / T.  The gradient then needs no cross sum; the
// forward KL's value, sum q (log q - log pT) (q, pT: the teacher's and the
// student's softmax at T), is summed as the pass goes and added to the row's
// losses after it, and the from-distribution CE is that plus the teacher's
// entropy (from its records).  Reverse KL is not covered: its
// coefficient needs the cross sum sum pT (log pT - log q) before the pass.
//
// Four warps per row, each a quarter of its words (a unit), units strided
// over the grid:
//   merge     the row's four warps merge a quarter of the tile records each
//             (running max, rescaled sums), exchange them through shared
//             memory, and each takes the 32 lane records through the row
//             epilogue shared with the other kernels (losses, coefficients);
//   gradient  the unit's words (and the teacher's) arrive through the warp's
//             own ring of 4 KB bulk copies, which runs ahead across units;
//             each lane computes the combined gradient of its 16-byte words
//             in fp32 and stores it once; the lane whose word holds the label
//             column patches that element before the store.
// Per-warp compensated sums of the row losses are added in warp order into
// one fp64 partial record per CTA, which the finalize kernel reduces.
#include "hl_rows16.cuh"

namespace hl {

constexpr int OP_THREADS = 256;
constexpr int OP_WARPS = OP_THREADS / 32;
constexpr int OP_PARTS = 4;           // warps per row, each a quarter of the row's words
constexpr int OP_SLOTS = 3;           // chunk slots of each warp's ring
constexpr int OP_SLOT_BYTES = 4096;   // a slot: 256 student words, or 128 student + 128 teacher
// dynamic shared memory: the warps' rings and their mbarriers
constexpr int OP_SMEM = OP_WARPS * OP_SLOTS * OP_SLOT_BYTES + OP_WARPS * OP_SLOTS * 8;

template <int FEAT>
__global__ void __launch_bounds__(OP_THREADS, 2)
    onepass_kernel16(const __grid_constant__ Params p, const float4* __restrict__ rs,
                     const float* __restrict__ rsT, const float4* __restrict__ rst, int NT) {
    using P16 = Pack16<__nv_bfloat16>;
    constexpr bool TEACH = (FEAT & F_TEACH) != 0;
    constexpr bool ENT = (FEAT & F_ENT) != 0;
    constexpr bool CAP = (FEAT & F_SOFTCAP) != 0;
    constexpr bool ENTG = ENT && (FEAT & F_ENTG) != 0;
    constexpr int EPW = 8;
    constexpr int CW = TEACH ? 128 : 256;  // words of each operand in a chunk
    constexpr int NF = TEACH ? 7 : 3;      // merged fields the part warps exchange
    static_assert(CW * 16 * (TEACH ? 2 : 1) == OP_SLOT_BYTES, "slot size");

    __shared__ float recs[OP_WARPS][32 * NREC];
    __shared__ float accs[OP_WARPS][2 * NACC];
    __shared__ RowLoss rls[OP_WARPS];
    __shared__ float xq[OP_WARPS];  // a unit's forward-KL sum, per warp
    extern __shared__ __align__(128) unsigned char ring_smem[];
    // the part warps' merged records, [part][field][lane], live in the
    // group's record area between the two merge barriers
    static_assert(OP_PARTS * NF * 32 <= OP_PARTS * 32 * NREC, "exchange area");

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t N = p.N, V = p.V;
    const int64_t nwords = V / EPW;
    const __nv_bfloat16* __restrict__ xg = static_cast<const __nv_bfloat16*>(p.x);
    const __nv_bfloat16* __restrict__ tg = static_cast<const __nv_bfloat16*>(p.t);
    __nv_bfloat16* gg = static_cast<__nv_bfloat16*>(p.g);
    const bool has_labels = p.labels != nullptr;
    const bool need_side = (p.flags & (L_GRPO | L_GRPO_STATS)) != 0;
    const float kk = *p.kscale;

    const float LOG2E = 1.4426950408889634f;
    const float LN2 = 0.6931471805599453f;
    const float s = p.s;
    const float K1 = s * LOG2E;
    const float invc = CAP ? 1.f / p.softcap : 0.f;
    const float A2 = CAP ? 2.f * LOG2E * invc : 0.f;
    const float Kc = CAP ? s * p.softcap * LOG2E : 0.f;
    const float invT = TEACH ? 1.f / p.T : 1.f;
    const float KT = LOG2E * invT;  // teacher: ut = t log2(e) / T
    // softcap: tanh by tiers, picked per chunk from the records' largest |x|:
    // A = degree-3 odd polynomial on |x| <= 0.45 c (only while Kc <= 48,
    // where its fit error stays below fp32 rounding of the exponentials),
    // B = degree 5 on |x| <= 0.8 c, X = ex2 + rcp (any x)
    const float XA = (CAP && Kc <= 48.f) ? HL_TANH_A_Y0 * p.softcap : 0.f;
    const float XB = CAP ? HL_TANH_B_Y0 * p.softcap : 0.f;
    // zs = x Q(x^2) with Q_k = s log2(e) C_k / c^(2k), formed in double
    f2 QA[4], QB[6];
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
    // 1 - tanh^2 = 1 - (zs / Kc)^2 on the polynomial tiers (|tanh| <= 0.67)
    const f2 mKc2 = pk1(CAP ? -1.f / (Kc * Kc) : 0.f), one2 = pk1(1.f);
    const f2 K2 = pk1(K1), A22 = pk1(A2), Kc2 = pk1(Kc);
    const f2 invT2 = pk1(invT), KinvT2 = pk1(K1 * invT), KT2 = pk1(KT);
    auto zs1 = [&](float v, float* om) -> float {
        return CAP ? __fmul_rn(tanh_a2x_1(__fmul_rn(v, A2), om), Kc) : __fmul_rn(v, K1);
    };

    for (int i = lane; i < 2 * NACC; i += 32) accs[warp][i] = 0.f;

    const int64_t gw = int64_t(blockIdx.x) * OP_WARPS + warp;
    const int64_t nw = int64_t(gridDim.x) * OP_WARPS;
    const int64_t nunits = N * OP_PARTS;

    // This warp's ring: its units' words stream through OP_SLOTS chunks of
    // shared memory by bulk copies (lane 0 issues, an mbarrier per slot
    // counts the bytes), refilled as soon as the warp has used a chunk and
    // running on across units, so the copies OP_SLOTS chunks ahead are always
    // in flight whatever the arithmetic is doing.  A slot holds CW student
    // words and, with a teacher, the teacher's CW words behind them.
    unsigned char* ring = ring_smem + size_t(warp) * OP_SLOTS * OP_SLOT_BYTES;
    uint64_t* fullb =
        reinterpret_cast<uint64_t*>(ring_smem + size_t(OP_WARPS) * OP_SLOTS * OP_SLOT_BYTES) +
        warp * OP_SLOTS;
    auto unit_range = [&](int64_t uu, int64_t& rr, int64_t& b0, int64_t& b1) {
        rr = uu / OP_PARTS;
        const int pt = int(uu - rr * OP_PARTS);
        b0 = nwords * pt / OP_PARTS;
        b1 = nwords * (pt + 1) / OP_PARTS;
    };
    // the issuer's stream position (lane 0): unit iu, chunk ic of it
    int64_t iu = gw;
    int64_t ic = 0;
    auto issue_next = [&](int sl) {
        if (iu >= nunits) return;
        int64_t rr, b0, b1;
        unit_range(iu, rr, b0, b1);
        const int64_t c0 = b0 + ic * CW;
        const int64_t cw = (b1 - c0) < CW ? (b1 - c0) : CW;
        const uint32_t bar = smem_addr(&fullb[sl]);
        const uint32_t dst = smem_addr(ring + size_t(sl) * OP_SLOT_BYTES);
        mbar_arrive_expect_tx(bar, uint32_t(cw * 16) * (TEACH ? 2u : 1u));
        bulk_g2s(dst, xg + rr * V + c0 * EPW, uint32_t(cw * 16), bar);
        if (TEACH) bulk_g2s(dst + CW * 16, tg + rr * V + c0 * EPW, uint32_t(cw * 16), bar);
        if (c0 + CW >= b1) {
            iu += nw;
            ic = 0;
        } else {
            ++ic;
        }
    };
    if (lane == 0) {
        for (int sl = 0; sl < OP_SLOTS; ++sl) mbar_init(smem_addr(&fullb[sl]), 1);
        fence_mbar_init();
        for (int sl = 0; sl < OP_SLOTS; ++sl) issue_next(sl);
    }
    __syncwarp();
    int slot = 0;
    uint32_t phase = 0;
    uint32_t lost = 0, lost_par = 0;
    // the next chunk of the stream: wait for it, hand back its base
    auto acquire = [&]() -> const unsigned char* {
        if (!mbar_wait_bounded(smem_addr(&fullb[slot]), phase, p.wait_ns)) {
            lost |= 1u << slot;
            lost_par = (lost_par & ~(1u << slot)) | (phase << slot);
            if (lane == 0) atomicOr(p.err, E_TIMEOUT);
        }
        return ring + size_t(slot) * OP_SLOT_BYTES;
    };
    // the warp is done with the chunk: refill its slot, step the ring
    auto release = [&]() {
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async();
            issue_next(slot);
        }
        if (++slot == OP_SLOTS) {
            slot = 0;
            phase ^= 1u;
        }
    };
    // the row's four warps (warps 0-3 or 4-7 of the CTA) take the same rows
    // in the same iterations: a named barrier of the four orders their
    // exchanges
    const uint32_t gbar = 1 + (warp >> 2);
    auto group_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(gbar) : "memory"); };
    float* mg = recs[(warp / OP_PARTS) * OP_PARTS];  // [part][field][lane]

    // unit u: row u / OP_PARTS, part u % OP_PARTS (a range of the row's words);
    // every part merges the row's records itself, part 0 adds the row's losses
    for (int64_t u = gw; u < nunits; u += nw) {
        const int64_t r = u / OP_PARTS;
        const int part = int(u - r * OP_PARTS);
        const int64_t wb = nwords * part / OP_PARTS, we = nwords * (part + 1) / OP_PARTS;
        const int64_t nch = (we - wb + CW - 1) / CW;
        int64_t y = 0;
        float old_lp = 0.f, adv = 0.f;
        if (lane == 0) {
            if (has_labels) y = p.labels[r];
            if (need_side) {
                old_lp = p.old_lp[r];
                adv = p.adv[r];
            }
        }
        // every lane derives the row's coefficients itself: all need the side inputs
        y = __shfl_sync(0xffffffffu, y, 0);
        old_lp = __shfl_sync(0xffffffffu, old_lp, 0);
        adv = __shfl_sync(0xffffffffu, adv, 0);
        const bool valid = !has_labels || (y >= 0 && y < V);
        if (has_labels && y >= V && lane == 0 && part == 0) atomicOr(p.err, E_LABEL);
        __nv_bfloat16* grow = gg != nullptr ? gg + r * V : nullptr;
        if (!valid) {  // a masked row: exact +0 (kept when accumulating); its chunks pass by
            if (lane == 0 && part == 0) write_row_zero(p, r);
            if (grow != nullptr && !p.accumulate)
                for (int64_t w = wb + lane; w < we; w += 32)
                    *reinterpret_cast<uint4*>(grow + w * EPW) = make_uint4(0, 0, 0, 0);
            for (int64_t c = 0; c < nch; ++c) {
                acquire();
                release();
            }
            continue;
        }

        // ---- merge the tiles' records: part warp pt, lane k takes tiles
        // pt 32 + k + 128 j (four tiles' loads in flight per lane), then lane
        // k of every part warp merges the four parts' records of lane k ----
        // student (M, S, E; S_T at the temperature), teacher (Mu, Sq, Eq)
        float M = -CUDART_INF_F, S = 0.f, E = 0.f, ST = 0.f, Mu = -CUDART_INF_F, Sq = 0.f,
              Eq = 0.f;
        auto merge_s = [&](float qm, float qs, float qe, float qt) {
            if (!(qs > 0.f)) return;
            if (qm > M) {
                const float d = M == -CUDART_INF_F ? 0.f : M - qm;  // <= 0
                const float al = exp2f(d);
                if (ENT) E = al * (E + d * S) + qe;
                S = al * S + qs;
                if (TEACH) ST = exp2f(d * invT) * ST + qt;
                M = qm;
            } else {
                const float d = qm - M;
                const float al = exp2f(d);
                if (ENT) E += al * (qe + d * qs);
                S += al * qs;
                if (TEACH) ST += exp2f(d * invT) * qt;
            }
        };
        auto merge_t = [&](float qm, float qs, float qe) {
            if (!(qs > 0.f)) return;
            if (qm > Mu) {
                const float d = Mu == -CUDART_INF_F ? 0.f : Mu - qm;  // <= 0
                const float al = exp2f(d);
                Eq = al * (Eq + d * Sq) + qe;
                Sq = al * Sq + qs;
                Mu = qm;
            } else {
                const float d = qm - Mu;
                const float al = exp2f(d);
                Eq += al * (qe + d * qs);
                Sq += al * qs;
            }
        };
        const float4* rrow = rs + r * NT;
        const float* trow = TEACH && rsT != nullptr ? rsT + r * NT : nullptr;
        const float4* urow = TEACH ? rst + r * NT : nullptr;
        for (int tb = part * 32 + lane; tb < NT; tb += 4 * 128) {
            float4 q[4], qu[4];
            float qt[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool in = tb + 128 * j < NT;
                q[j] = in ? rrow[tb + 128 * j] : make_float4(0.f, 0.f, 0.f, 0.f);
                if (TEACH) {
                    qu[j] = in ? urow[tb + 128 * j] : make_float4(0.f, 0.f, 0.f, 0.f);
                    qt[j] = in && trow != nullptr ? trow[tb + 128 * j] : q[j].y;  // T = 1: S
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                merge_s(q[j].x, q[j].y, q[j].z, TEACH ? qt[j] : 0.f);
                if (TEACH) merge_t(qu[j].x, qu[j].y, qu[j].z);
            }
        }
        float zy = 0.f, hasy = 0.f;
        if (lane == 0 && has_labels) {
            zy = zs1(P16::to_f(reinterpret_cast<const uint16_t*>(xg)[r * V + y]), nullptr);
            hasy = 1.f;
        }
        {
            float* m = mg + part * NF * 32 + lane;
            m[0] = M;
            m[32] = S;
            m[64] = E;
            if (TEACH) {
                m[96] = ST;
                m[128] = Mu;
                m[160] = Sq;
                m[192] = Eq;
            }
        }
        // all four warps have read the label logit and stored their records
        // before any of them writes the gradient (in place, one of them
        // overwrites the label logit) or the merged records (next)
        group_sync();
        M = -CUDART_INF_F;
        S = E = ST = Sq = Eq = 0.f;
        Mu = -CUDART_INF_F;
#pragma unroll
        for (int pt = 0; pt < OP_PARTS; ++pt) {
            const float* m = mg + pt * NF * 32 + lane;
            merge_s(m[0], m[32], m[64], TEACH ? m[96] : 0.f);
            if (TEACH) merge_t(m[128], m[160], m[192]);
        }
        // all have read the exchanged records before the area takes the
        // lane records below
        group_sync();
        float* rec = recs[warp] + lane * NREC;
        rec[R_ZM] = M;
        rec[R_UM] = Mu;
        rec[R_S] = S;
        rec[R_E] = E;
        rec[R_ST] = ST;
        rec[R_SQ] = Sq;
        rec[R_EQ] = Eq;
        rec[R_XP] = 0.f;  // the forward KL comes from the pass (below)
        rec[R_Y] = 0.f;
        rec[R_ZY] = zy;
        rec[R_HASY] = hasy;
        __syncwarp();
        RowCoef k = row_epilogue16<TEACH, false, ENT, CAP, true>(
            p, recs[warp], 32, false, old_lp, adv, accs[warp], lane, r, kk, &rls[warp]);
        if (p.tok != nullptr) {
            // a per-token coefficient c = d(total)/d(log p(label)) (GSPO's):
            // c (delta_label - p), scaled like every coefficient
            const float c = p.tok[r] * p.s;
            k.pc -= c;
            k.bc -= c;
        }
        // all have read their lane records before the next row's exchange
        // reuses the area
        group_sync();
        if (!TEACH && lane == 0 && part == 0) row_accumulate(p, rls[warp], accs[warp], r);
        if (!TEACH && grow == nullptr) {
            for (int64_t c = 0; c < nch; ++c) {
                acquire();
                release();
            }
            continue;
        }

        // ---- the gradient, one read and one write of the row ----
        const ShiftCoef h = shift_coefs(k, ENTG);
        const f2 nlse2 = pk1(h.nlse), pc2 = pk1(h.pc), ps2 = pk1(h.ps);
        const f2 nlseT2 = pk1(h.nlseT), nlsq2 = pk1(h.nlsq), tc2 = pk1(h.tc), qc2 = pk1(h.qc);
        const int64_t ywd = has_labels ? y / EPW : -1;  // the label's word
        const int iyw = has_labels ? int(y - ywd * EPW) : 0;
        // the forward KL's sum over this unit, in units of 2^sg (the
        // exponent shift shared by every exponential): B1 = sum 2^sg q
        // (log2 q - log2 pT)
        f2 B1 = pk1(0.f);
        // softcap: the tier of chunk c of this unit (c < 32; later chunks take
        // tier X): lane c takes the largest |x| of the tiles the chunk spans
        uint32_t mA = 0u, mB = 0u;
        if (CAP) {
            float cx = 0.f;
            if (lane < nch) {
                const int64_t c0 = wb + int64_t(lane) * CW;
                const int64_t c1 = c0 + CW < we ? c0 + CW : we;
                const int64_t t0 = c0 / 32, t1 = (c1 - 1) / 32;  // 32 words a tile
                const float* xr = reinterpret_cast<const float*>(rrow) + 3;
#pragma unroll
                for (int i = 0; i <= CW / 32; ++i)
                    if (t0 + i <= t1) cx = fmaxf(cx, xr[4 * (t0 + i)]);
            }
            mA = __ballot_sync(0xffffffffu, cx <= XA);
            mB = __ballot_sync(0xffffffffu, cx <= XB);
        }
        // one word's gradient in tier TI (-1: no softcap); b: the teacher's
        // word; live: a word of the unit (the cross sums take only those)
        auto word = [&](const uint4& a, const uint4& b, const uint4& ow, bool live,
                        auto tierc) -> uint4 {
            constexpr int TI = decltype(tierc)::value;
            const uint32_t xa[4] = {a.x, a.y, a.z, a.w};
            const uint32_t ta[4] = {b.x, b.y, b.z, b.w};
            const uint32_t oa[4] = {ow.x, ow.y, ow.z, ow.w};
            uint32_t out[4];
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const f2 xv = P16::unpack(xa[kq]);
                f2 arg, argT = pk1(0.f), omt = one2;
                if constexpr (TI < 0) {
                    arg = fma2(xv, K2, nlse2);
                    if (TEACH) argT = fma2(xv, KinvT2, nlseT2);
                } else if constexpr (TI <= 1) {
                    const f2 u = mul2(xv, xv);
                    f2 q;
                    if constexpr (TI == 0) {
                        q = fma2(u, QA[3], QA[2]);
                        q = fma2(q, u, QA[1]);
                        q = fma2(q, u, QA[0]);
                    } else {
                        q = fma2(u, QB[5], QB[4]);
                        q = fma2(q, u, QB[3]);
                        q = fma2(q, u, QB[2]);
                        q = fma2(q, u, QB[1]);
                        q = fma2(q, u, QB[0]);
                    }
                    const f2 zs = mul2(xv, q);
                    omt = fma2(zs, mul2(zs, mKc2), one2);
                    arg = add2(zs, nlse2);
                    if (TEACH) argT = fma2(zs, invT2, nlseT2);
                } else {
                    const TanhD2 td = tanh_from_ex2_arg(mul2(xv, A22));
                    omt = td.omt;
                    const f2 zs = mul2(td.th, Kc2);
                    arg = add2(zs, nlse2);
                    if (TEACH) argT = fma2(zs, invT2, nlseT2);
                }
                f2 g = mul2(ex2p(arg), ENTG ? fma2(ps2, arg, pc2) : pc2);
                if (TEACH) {
                    const f2 argq = fma2(P16::unpack(ta[kq]), KT2, nlsq2);
                    const f2 pT = ex2p(argT), q = ex2p(argq);
                    g = fma2(pT, tc2, g);
                    g = fma2(q, qc2, g);
                    if (live) B1 = fma2(q, sub2(argq, argT), B1);
                }
                const f2 gw = CAP ? mul2(g, omt) : g;
                out[kq] = P16::pack(p.accumulate ? add2(P16::unpack(oa[kq]), gw) : gw);
            }
            return make_uint4(out[0], out[1], out[2], out[3]);
        };
        // the label column's element again, with the label term (halves
        // picked by selects, so the words stay in registers)
        auto patch = [&](const uint4& o, const uint4& a, const uint4& b,
                         const uint4& ow) -> uint4 {
            const uint32_t xa[4] = {a.x, a.y, a.z, a.w};
            const uint32_t ta[4] = {b.x, b.y, b.z, b.w};
            const uint32_t oa[4] = {ow.x, ow.y, ow.z, ow.w};
            uint32_t out[4] = {o.x, o.y, o.z, o.w};
            const int qy = iyw >> 1, sh = (iyw & 1) * 16;
            uint32_t xw = xa[0], tw = ta[0], owd = oa[0];
#pragma unroll
            for (int kq = 1; kq < 4; ++kq)
                if (kq == qy) {
                    xw = xa[kq];
                    tw = ta[kq];
                    owd = oa[kq];
                }
            const float xv1 = P16::to_f(uint16_t(xw >> sh));
            float om1 = 1.f;
            const float zs = zs1(xv1, &om1);
            const float arg = zs + h.nlse;
            float g1 = ex2f(arg) * (ENTG ? fmaf(h.ps, arg, h.pc) : h.pc);
            if (TEACH) {
                g1 = fmaf(ex2f(fmaf(zs, invT, h.nlseT)), h.tc, g1);
                g1 = fmaf(ex2f(fmaf(P16::to_f(uint16_t(tw >> sh)), KT, h.nlsq)), h.qc, g1);
            }
            g1 -= k.bc;
            if (CAP) g1 *= om1;
            if (p.accumulate) g1 += P16::to_f(uint16_t(owd >> sh));
            const uint32_t hv = uint32_t(P16::from_f(g1)) << sh;
            const uint32_t keep = sh ? 0x0000ffffu : 0xffff0000u;
#pragma unroll
            for (int kq = 0; kq < 4; ++kq)
                if (kq == qy) out[kq] = (out[kq] & keep) | hv;
            return make_uint4(out[0], out[1], out[2], out[3]);
        };
        // one chunk from the ring: CW / 32 words a lane, unrolled; the words
        // past a short chunk's end are computed and neither stored nor summed
        // (with a teacher a full chunk, the common case, tests no word)
        const bool store = grow != nullptr;
        auto chunk = [&](const unsigned char* sb, __nv_bfloat16* gc, int cw, int jy, auto tierc,
                         auto fullc) {
            constexpr bool FULL = decltype(fullc)::value;
#pragma unroll
            for (int i = 0; i < CW / 32; ++i) {
                const int j = lane + 32 * i;
                const bool in = FULL || j < cw;
                const uint4 a = *reinterpret_cast<const uint4*>(sb + size_t(j) * 16);
                uint4 b = make_uint4(0, 0, 0, 0);
                if (TEACH) b = *reinterpret_cast<const uint4*>(sb + CW * 16 + size_t(j) * 16);
                uint4 ow = make_uint4(0, 0, 0, 0);
                if (p.accumulate && in) ow = *reinterpret_cast<const uint4*>(gc + size_t(j) * EPW);
                uint4 o = word(a, b, ow, in, tierc);
                if (j == jy) o = patch(o, a, b, ow);
                if (store && in) *reinterpret_cast<uint4*>(gc + size_t(j) * EPW) = o;
            }
        };
        // (the split pays only where a word's test guards the cross sum: with
        // a teacher; without, the doubled code measured slower)
        auto chunk_t = [&](const unsigned char* sb, __nv_bfloat16* gc, int cw, int jy,
                           auto tierc) {
            if (TEACH && cw == CW) chunk(sb, gc, cw, jy, tierc, std::true_type{});
            else chunk(sb, gc, cw, jy, tierc, std::false_type{});
        };
        for (int64_t c = 0; c < nch; ++c) {
            const unsigned char* sb = acquire();
            const int64_t c0 = wb + c * CW;
            const int cw = int((we - c0) < CW ? (we - c0) : CW);
            const int jy = (ywd >= c0 && ywd < c0 + cw) ? int(ywd - c0) : -1;
            __nv_bfloat16* gc = store ? grow + c0 * EPW : nullptr;
            if (!CAP) {
                chunk_t(sb, gc, cw, jy, std::integral_constant<int, -1>{});
            } else {
                const bool inA = c < 32 && ((mA >> c) & 1u), inB = c < 32 && ((mB >> c) & 1u);
                if (inA) chunk_t(sb, gc, cw, jy, std::integral_constant<int, 0>{});
                else if (inB) chunk_t(sb, gc, cw, jy, std::integral_constant<int, 1>{});
                else chunk_t(sb, gc, cw, jy, std::integral_constant<int, 2>{});
            }
            release();
        }
        if (TEACH) {
            // the row's distillation values: forward KL = ln2 sum q (log2 q -
            // log2 pT) from the four warps' sums; the epilogue's values, with
            // the cross sum left out, differ by the teacher's entropy
            // (from-distribution CE = forward KL + H(q)), which holds for the
            // true values as well
            float b1 = hsum(B1);
#pragma unroll
            for (int o = 16; o; o >>= 1) b1 += __shfl_xor_sync(0xffffffffu, b1, o);
            if (lane == 0) xq[warp] = b1;
            group_sync();
            if (lane == 0 && part == 0) {
                float s1 = 0.f;
                for (int pt = 0; pt < OP_PARTS; ++pt) s1 += xq[warp + pt];
                const float sg = rintf(h.nlsq + k.lsq2);  // the shift: nlsq = sg - lsq2
                const float sc = __uint_as_float(uint32_t(127 - int(sg)) << 23);  // 2^-sg
                const float fkl = LN2 * s1 * sc;
                rls[warp].dce = fkl + (rls[warp].dce - rls[warp].fkl);
                rls[warp].fkl = fkl;
                row_accumulate(p, rls[warp], accs[warp], r);
            }
        }
    }

    // a slot whose wait gave up may still receive its copy: wait once more
    // (bounded) before the CTA's shared memory goes away
    if (lost && lane == 0)
        for (int b = 0; b < OP_SLOTS; ++b)
            if (lost & (1u << b))
                (void)mbar_wait_bounded(smem_addr(&fullb[b]), (lost_par >> b) & 1u, p.wait_ns);

    // the warps' sums, in warp order, into the CTA's fp64 partial record
    __syncthreads();
    if (threadIdx.x < NACC) {
        double t = 0.0;
        for (int w = 0; w < OP_WARPS; ++w)
            t += double(accs[w][threadIdx.x]) - double(accs[w][NACC + threadIdx.x]);
        p.partials[size_t(blockIdx.x) * NACC + threadIdx.x] = t;
    }
}

#define HL_CASE(F) \
    case F: return reinterpret_cast<const void*>(&onepass_kernel16<F>);

const void* onepass_kernel_bf16(int feat) {
    switch (feat) {
        HL_CASE(0)
        HL_CASE(F_ENT)
        HL_CASE(F_ENT | F_ENTG)
        HL_CASE(F_SOFTCAP)
        HL_CASE(F_SOFTCAP | F_ENT)
        HL_CASE(F_SOFTCAP | F_ENT | F_ENTG)
        HL_CASE(F_TEACH)
        HL_CASE(F_TEACH | F_ENT)
        HL_CASE(F_TEACH | F_ENT | F_ENTG)
        HL_CASE(F_TEACH | F_SOFTCAP)
        HL_CASE(F_TEACH | F_SOFTCAP | F_ENT)
        HL_CASE(F_TEACH | F_SOFTCAP | F_ENT | F_ENTG)
        default: return nullptr;
    }
}

#undef HL_CASE

int onepass_smem_bytes() { return OP_SMEM; }

}  // namespace hl
