// hl_gspo.cu -- GSPO's segment seam (headloss_gspo_seam in include/headloss.h).
//
// GSPO is the sequence-level clipped policy objective: per segment i of
// valid rows T_i (L_i of them), the ratio s_i = exp((1/L_i) sum_t (lp_t -
// old_t)) -- the geometric mean of the token ratios -- and the objective
// min(s_i A_i, clip(s_i, 1 - eps, 1 + eps) A_i), A_i the mean advantage of
// the segment; the loss is minus its mean over the G segments that hold a
// valid row.  Its gradient reaches each row only through the row's label
// log-prob, with coefficient
//   c_t = d(weight * grad_scale * loss) / d lp_t = -weight grad_scale A_i s_i act_i / (G L_i)
// (act_i: the unclipped branch is the smaller objective, ties included).
// The seam runs between a forward call that produced lp (new_logprobs of
// headloss_forward_backward_ext) and the backward call that superposes c on
// the label column (token_coeff): ServiceNow Fast-LLM PR #558, "Design"
// (the GSPO seam hands the kernel a per-token coefficient) and PR #549,
// "Loss coverage" (GSPO's per-segment seam).
//
// One block of 1024 threads, fp64 throughout (O(N) work).  Warp w takes
// segments w, w + 32, ...: pass 1 forms each segment's sums and the warp's
// partial sums over its segments; the block adds the 32 partials in warp
// order (the result does not depend on timing); pass 2 recomputes each
// segment's values with the same arithmetic and writes its rows'
// coefficients.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "headloss.h"

namespace hl_gspo {

constexpr int THREADS = 1024;
constexpr int WARPS = THREADS / 32;

struct Seg {
    double L, s, A, obj;
    bool act, clipped;
};

// The sums of segment i over its valid rows, in every lane of the warp.
__device__ Seg segment(const float* lp, const float* old, const float* adv, const int64_t* labels,
                       int64_t N, int64_t V, const int64_t* off, int i, double eps, int lane) {
    int64_t a = off[i], b = off[i + 1];
    a = a < 0 ? 0 : (a > N ? N : a);
    b = b < a ? a : (b > N ? N : b);
    double L = 0.0, d = 0.0, A = 0.0;
    for (int64_t t = a + lane; t < b; t += 32) {
        const int64_t y = labels[t];
        if (y < 0 || y >= V) continue;
        L += 1.0;
        d += double(lp[t]) - double(old[t]);
        A += double(adv[t]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        L += __shfl_xor_sync(0xffffffffu, L, o);
        d += __shfl_xor_sync(0xffffffffu, d, o);
        A += __shfl_xor_sync(0xffffffffu, A, o);
    }
    Seg sg{L, 0.0, 0.0, 0.0, false, false};
    if (L > 0.0) {
        sg.s = exp(d / L);
        sg.A = A / L;
        double sc = sg.s < 1.0 - eps ? 1.0 - eps : sg.s;
        sc = sc > 1.0 + eps ? 1.0 + eps : sc;
        const double unc = sg.s * sg.A, clp = sc * sg.A;
        sg.obj = unc < clp ? unc : clp;
        sg.act = unc <= clp || (sg.s >= 1.0 - eps && sg.s <= 1.0 + eps);
        sg.clipped = fabs(sg.s - 1.0) > eps;
    }
    return sg;
}

__global__ void __launch_bounds__(THREADS) gspo_seam_kernel(
    const float* lp, const float* old, const float* adv, const int64_t* labels, int64_t N,
    int64_t V, const int64_t* off, int n_seg, double eps, double wg, float* coeff, float* out) {
    __shared__ double part[WARPS][4];  // G, sum obj, sum s, clipped
    __shared__ double tot[4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    double g = 0.0, so = 0.0, ss = 0.0, sc = 0.0;
    for (int i = warp; i < n_seg; i += WARPS) {
        const Seg sg = segment(lp, old, adv, labels, N, V, off, i, eps, lane);
        if (sg.L > 0.0) {
            g += 1.0;
            so += sg.obj;
            ss += sg.s;
            sc += sg.clipped ? 1.0 : 0.0;
        }
    }
    if (lane == 0) {
        part[warp][0] = g;
        part[warp][1] = so;
        part[warp][2] = ss;
        part[warp][3] = sc;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        double t = 0.0;
        for (int w = 0; w < WARPS; ++w) t += part[w][threadIdx.x];
        tot[threadIdx.x] = t;
    }
    __syncthreads();
    const double G = tot[0];
    if (threadIdx.x == 0) {
        out[0] = G > 0.0 ? float(-tot[1] / G) : 0.f;
        out[1] = G > 0.0 ? float(tot[2] / G) : 0.f;
        out[2] = G > 0.0 ? float(tot[3] / G) : 0.f;
        out[3] = float(G);
    }
    // pass 2: the rows' coefficients (rows outside every segment get 0 below)
    for (int i = warp; i < n_seg; i += WARPS) {
        const Seg sg = segment(lp, old, adv, labels, N, V, off, i, eps, lane);
        int64_t a = off[i], b = off[i + 1];
        a = a < 0 ? 0 : (a > N ? N : a);
        b = b < a ? a : (b > N ? N : b);
        const double c = (sg.L > 0.0 && sg.act) ? -wg * sg.A * sg.s / (G * sg.L) : 0.0;
        for (int64_t t = a + lane; t < b; t += 32) {
            const int64_t y = labels[t];
            coeff[t] = (y < 0 || y >= V) ? 0.f : float(c);
        }
    }
}

// Rows before the first segment or after the last one carry no GSPO term.
__global__ void gspo_zero_kernel(float* coeff, int64_t N) {
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < N;
         t += int64_t(gridDim.x) * blockDim.x)
        coeff[t] = 0.f;
}

}  // namespace hl_gspo

extern "C" int headloss_gspo_seam(const float* new_logprobs, const float* old_logprobs,
                                  const float* advantages, const int64_t* labels, int64_t N,
                                  int64_t V, const int64_t* seg_offsets, int n_seg, float clip_eps,
                                  float weight, float grad_scale, float* token_coeff,
                                  float* scalars_out, headloss_stream_t stream) {
    using namespace hl_gspo;
    if (N < 0 || V < 1 || n_seg < 1) return HEADLOSS_ERR_ARG;
    if (!(clip_eps >= 0.f) || !isfinite(clip_eps) || !isfinite(weight) || !isfinite(grad_scale))
        return HEADLOSS_ERR_ARG;
    if (!seg_offsets || !scalars_out) return HEADLOSS_ERR_ARG;
    if (N > 0 && (!new_logprobs || !old_logprobs || !advantages || !labels || !token_coeff))
        return HEADLOSS_ERR_ARG;
    const uintptr_t a4 = reinterpret_cast<uintptr_t>(new_logprobs) |
                         reinterpret_cast<uintptr_t>(old_logprobs) |
                         reinterpret_cast<uintptr_t>(advantages) |
                         reinterpret_cast<uintptr_t>(token_coeff) |
                         reinterpret_cast<uintptr_t>(scalars_out);
    const uintptr_t a8 = reinterpret_cast<uintptr_t>(labels) |
                         reinterpret_cast<uintptr_t>(seg_offsets);
    if ((a4 & 3u) || (a8 & 7u)) return HEADLOSS_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N > 0) gspo_zero_kernel<<<64, 256, 0, s>>>(token_coeff, N);
    gspo_seam_kernel<<<1, THREADS, 0, s>>>(new_logprobs, old_logprobs, advantages, labels, N, V,
                                           seg_offsets, n_seg, double(clip_eps),
                                           double(weight) * double(grad_scale), token_coeff,
                                           scalars_out);
    return cudaGetLastError() == cudaSuccess ? HEADLOSS_OK : HEADLOSS_ERR_CUDA;
}
