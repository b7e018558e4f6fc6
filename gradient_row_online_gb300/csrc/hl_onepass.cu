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
// record (m2, S, E) of zs = s c tanh(x / c) log2(e) (c = 0: s x log2(e)):
// m2 = max zs, S = sum 2^(zs - m2), E = sum 2^(zs - m2) (zs - m2).  These
// cover every label-based loss (CE, z-loss, GRPO and its statistics,
// entropy); the distillation losses pair the row with a teacher row element
// by element and are not supported here.
//
// One warp per row, rows strided over the grid:
//   merge     lane k merges the records of tiles k, k + 32, ... (running max,
//             rescaled sums); the 32 lane records go through the row epilogue
//             shared with the other kernels (losses, coefficients);
//   gradient  each lane streams 16-byte words of the row (a warp reads and
//             writes 512 contiguous bytes per step), computes the combined
//             gradient in fp32 and writes it once; the lane whose word holds
//             the label column patches that element before the store.
// Per-warp compensated sums of the row losses are added in warp order into
// one fp64 partial record per CTA, which the finalize kernel reduces.
#include "hl_rows16.cuh"

namespace hl {

constexpr int OP_THREADS = 256;
constexpr int OP_WARPS = OP_THREADS / 32;
constexpr int OP_PARTS = 4;   // warps per row, each a quarter of the row's words
constexpr int OP_UNROLL = 4;  // words per lane in flight

template <int FEAT>
__global__ void __launch_bounds__(OP_THREADS, 3) onepass_kernel16(const __grid_constant__ Params p,
                                                               const float4* __restrict__ rs,
                                                               int NT) {
    using P16 = Pack16<__nv_bfloat16>;
    constexpr bool ENT = (FEAT & F_ENT) != 0;
    constexpr bool CAP = (FEAT & F_SOFTCAP) != 0;
    constexpr bool ENTG = ENT && (FEAT & F_ENTG) != 0;
    constexpr int EPW = 8;

    __shared__ float recs[OP_WARPS][32 * NREC];
    __shared__ float accs[OP_WARPS][2 * NACC];
    __shared__ RowLoss rls[OP_WARPS];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t N = p.N, V = p.V;
    const int64_t nwords = V / EPW;
    const __nv_bfloat16* __restrict__ xg = static_cast<const __nv_bfloat16*>(p.x);
    __nv_bfloat16* gg = static_cast<__nv_bfloat16*>(p.g);
    const bool has_labels = p.labels != nullptr;
    const bool need_side = (p.flags & (L_GRPO | L_GRPO_STATS)) != 0;
    const float kk = *p.kscale;

    const float LOG2E = 1.4426950408889634f;
    const float s = p.s;
    const float K1 = s * LOG2E;
    const float invc = CAP ? 1.f / p.softcap : 0.f;
    const float A2 = CAP ? 2.f * LOG2E * invc : 0.f;
    const float Kc = CAP ? s * p.softcap * LOG2E : 0.f;
    const float XP = CAP ? HL_TANH_POLY_Y0 * p.softcap : 0.f;  // polynomial range on |x|
    const f2 K2 = pk1(K1), A22 = pk1(A2), Kc2 = pk1(Kc), invc2 = pk1(invc);
    auto zs1 = [&](float v, float* om) -> float {
        return CAP ? __fmul_rn(tanh_a2x_1(__fmul_rn(v, A2), om), Kc) : __fmul_rn(v, K1);
    };

    for (int i = lane; i < 2 * NACC; i += 32) accs[warp][i] = 0.f;
    __syncwarp();

    const int64_t gw = int64_t(blockIdx.x) * OP_WARPS + warp;
    const int64_t nw = int64_t(gridDim.x) * OP_WARPS;
    // unit u: row u / OP_PARTS, part u % OP_PARTS (a range of the row's words);
    // every part merges the row's records itself, part 0 adds the row's losses
    for (int64_t u = gw; u < N * OP_PARTS; u += nw) {
        const int64_t r = u / OP_PARTS;
        const int part = int(u - r * OP_PARTS);
        const int64_t wb = nwords * part / OP_PARTS, we = nwords * (part + 1) / OP_PARTS;
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
        if (!valid) {  // a masked row: exact +0 (kept when accumulating)
            if (lane == 0 && part == 0) write_row_zero(p, r);
            if (grow != nullptr && !p.accumulate)
                for (int64_t w = wb + lane; w < we; w += 32)
                    *reinterpret_cast<uint4*>(grow + w * EPW) = make_uint4(0, 0, 0, 0);
            continue;
        }

        // ---- merge the tiles' records: lane k takes tiles k, k + 32, ... ----
        float M = -CUDART_INF_F, S = 0.f, E = 0.f;
        const float4* rrow = rs + r * NT;
        for (int t = lane; t < NT; t += 32) {
            const float4 q = rrow[t];
            if (!(q.y > 0.f)) continue;
            if (q.x > M) {
                const float d = M == -CUDART_INF_F ? 0.f : M - q.x;  // <= 0
                const float al = exp2f(d);
                if (ENT) E = al * (E + d * S) + q.z;
                S = al * S + q.y;
                M = q.x;
            } else {
                const float d = q.x - M;
                const float al = exp2f(d);
                if (ENT) E += al * (q.z + d * q.y);
                S += al * q.y;
            }
        }
        float zy = 0.f, hasy = 0.f;
        if (lane == 0 && has_labels) {
            zy = zs1(P16::to_f(reinterpret_cast<const uint16_t*>(xg)[r * V + y]), nullptr);
            hasy = 1.f;
        }
        float* rec = recs[warp] + lane * NREC;
        rec[R_ZM] = M;
        rec[R_UM] = 0.f;
        rec[R_S] = S;
        rec[R_E] = E;
        rec[R_ST] = 0.f;
        rec[R_SQ] = 0.f;
        rec[R_EQ] = 0.f;
        rec[R_XP] = 0.f;
        rec[R_Y] = 0.f;
        rec[R_ZY] = zy;
        rec[R_HASY] = hasy;
        __syncwarp();
        const RowCoef k = row_epilogue16<false, false, ENT, CAP, true>(
            p, recs[warp], 32, false, old_lp, adv, accs[warp], lane, r, kk, &rls[warp]);
        __syncwarp();
        if (lane == 0 && part == 0) row_accumulate(p, rls[warp], accs[warp], r);
        if (grow == nullptr) continue;

        // ---- the gradient, one read and one write of the row ----
        const ShiftCoef h = shift_coefs(k, ENTG);
        const f2 nlse2 = pk1(h.nlse), pc2 = pk1(h.pc), ps2 = pk1(h.ps);
        const int64_t ywd = has_labels ? y / EPW : -1;
        // one word of the row: its gradient, the label element patched
        auto word = [&](int64_t w, const uint4& a, const uint4& ow) -> uint4 {
            const uint32_t xa[4] = {a.x, a.y, a.z, a.w};
            const uint32_t oa[4] = {ow.x, ow.y, ow.z, ow.w};
            bool poly = true;
            if (CAP) {
                const uint32_t am = P16::absmax2(P16::absmax2(a.x, a.y), P16::absmax2(a.z, a.w));
                float ca, cb;
                upk(P16::unpack(am), ca, cb);
                poly = fmaxf(fabsf(ca), fabsf(cb)) <= XP;
            }
            uint32_t out[4];
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const f2 xv = P16::unpack(xa[kq]);
                f2 arg, omt = pk1(1.f);
                if (CAP) {
                    const TanhD2 td =
                        poly ? tanh_poly2(mul2(xv, invc2)) : tanh_from_ex2_arg(mul2(xv, A22));
                    arg = fma2(td.th, Kc2, nlse2);
                    omt = td.omt;
                } else {
                    arg = fma2(xv, K2, nlse2);
                }
                const f2 g = mul2(ex2p(arg), ENTG ? fma2(ps2, arg, pc2) : pc2);
                const f2 gw = CAP ? mul2(g, omt) : g;
                out[kq] = P16::pack(p.accumulate ? add2(P16::unpack(oa[kq]), gw) : gw);
            }
            if (w == ywd) {
                // the label column: its element again, with the label term
                // (halves picked by selects, so the words stay in registers)
                const int iy = int(y - w * EPW), qy = iy >> 1, sh = (iy & 1) * 16;
                uint32_t xw = xa[0], owd = oa[0];
#pragma unroll
                for (int kq = 1; kq < 4; ++kq)
                    if (kq == qy) {
                        xw = xa[kq];
                        owd = oa[kq];
                    }
                const float xv1 = P16::to_f(uint16_t(xw >> sh));
                float om1 = 1.f;
                const float zs = zs1(xv1, &om1);
                const float arg = zs + h.nlse;
                float g1 = ex2f(arg) * (ENTG ? fmaf(h.ps, arg, h.pc) : h.pc) - k.bc;
                if (CAP) g1 *= om1;
                if (p.accumulate) g1 += P16::to_f(uint16_t(owd >> sh));
                const uint32_t hv = uint32_t(P16::from_f(g1)) << sh;
                const uint32_t keep = sh ? 0x0000ffffu : 0xffff0000u;
#pragma unroll
                for (int kq = 0; kq < 4; ++kq)
                    if (kq == qy) out[kq] = (out[kq] & keep) | hv;
            }
            return make_uint4(out[0], out[1], out[2], out[3]);
        };
        // OP_UNROLL words per lane per step: their loads are all in flight
        // before the first is used
        const __nv_bfloat16* xrow = xg + r * V;
        for (int64_t w0 = wb + lane; w0 < we; w0 += 32 * OP_UNROLL) {
            uint4 a[OP_UNROLL], ow[OP_UNROLL];
#pragma unroll
            for (int q = 0; q < OP_UNROLL; ++q) {
                const int64_t w = w0 + 32 * q;
                a[q] = make_uint4(0, 0, 0, 0);
                ow[q] = make_uint4(0, 0, 0, 0);
                if (w < we) {
                    a[q] = *reinterpret_cast<const uint4*>(xrow + w * EPW);
                    if (p.accumulate) ow[q] = *reinterpret_cast<const uint4*>(grow + w * EPW);
                }
            }
#pragma unroll
            for (int q = 0; q < OP_UNROLL; ++q) {
                const int64_t w = w0 + 32 * q;
                if (w < we) *reinterpret_cast<uint4*>(grow + w * EPW) = word(w, a[q], ow[q]);
            }
        }
    }

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
        default: return nullptr;
    }
}

#undef HL_CASE

}  // namespace hl
