// lmhead_tc.cu -- the LM-head GEMM in front of the loss, on the 5th-gen
// tensor cores: logits = hidden . weight^T (bf16 in, fp32 accumulation in
// TMEM, bf16 out) and, per (row, 256-column tile), the row statistics
// (max, sum of exp(x - max)) of the bf16-rounded logits.  It is the first
// building block of the fused LM head (the head GEMM whose output the loss
// consumes; tied embeddings and the LM head are PR #549 "Correctness" axes).
//
// A persistent kernel: one CTA per SM walks the 128 x 256 output tiles in a
// grouped order (GN column tiles at a time, every row tile within a group),
// so the weight panel of a group stays in L2 while the hidden rows stream.
// 192 threads:
//   warp 0: TMA producer (one thread), a 4-stage ring of hidden 128 x 64 and
//           weight 256 x 64 bf16 tiles, 128-byte swizzle
//   warp 1: TMEM allocation (all 512 columns: two 256-column accumulators)
//           and MMA issue (one thread): tcgen05.mma kind::f16, M = 128,
//           N = 256, K = 16, each stage committed to its "empty" barrier and
//           each tile to its accumulator's "full" barrier
//   warps 2..5: epilogue, one TMEM lane (= one tile row) per thread; while
//           they drain one accumulator the MMAs fill the other.  Each warp
//           stages 32 rows x 64 columns of bf16 at a time in shared memory
//           (128-byte swizzle, double-buffered) and writes them with a TMA
//           store, so global stores are whole 128-byte lines.
// Every wait is bounded by %globaltimer.  A wait that gives up sets bit 0 of
// *err and a shared abort flag; every role then stops issuing work, and the
// kernel waits (bounded) for the copies and MMAs it has issued before it
// frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "headloss.h"
#include "headloss_lmhead.h"

namespace hl_lmhead {

constexpr int BM = 128, BN = 256, BK = 64;  // BK bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int OUT_COLS = 64;                     // columns per staged store (128 bytes)
constexpr int OUT_BYTES = 32 * OUT_COLS * 2;     // 4 KB: 32 rows of one warp
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;              // two accumulators of BN columns
constexpr int GN = 16;                           // column tiles per group of the tile order
constexpr int RING_OFF = 0;
constexpr int OUT_OFF = STAGES * STAGE_BYTES;
constexpr int BAR_OFF = OUT_OFF + EPI_WARPS * 2 * OUT_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
constexpr unsigned long long WAIT_NS = 2000000000ull;
static_assert(SMEM_BYTES <= 232448, "shared memory");

__device__ __forceinline__ uint32_t su32(const void* p) {
    return uint32_t(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of parity `parity` of `bar`.  Returns false, without
// waiting further, once the kernel is aborting; gives up after WAIT_NS of
// wall time, raising *err and the abort flag.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                           int* err) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (gtimer() - t0 > WAIT_NS) {
            *abort = 1;
            atomicOr(err, 1);
            return false;
        }
    }
}
// The same, for the final drain: ignores the abort flag, bounded by time.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, int* err) {
    const uint64_t t0 = gtimer();
    while (!mbar_try(bar, parity))
        if (gtimer() - t0 > WAIT_NS) {
            atomicOr(err, 1);
            return;
        }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one committed store group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) |
           (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t instr_desc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
           (uint32_t(BM >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// 32 lanes x 32 columns of fp32 from TMEM: thread t gets lane (base lane + t),
// columns col .. col + 31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Output tile of position i in the grouped order: column tiles in groups of
// GN (the last group may be narrower), every row tile within a group.
__device__ __forceinline__ void tile_of(int i, int MT, int NT, int& m, int& n) {
    const int full = NT / GN;
    const int in_full = full * MT * GN;
    if (i < in_full) {
        const int g = i / (MT * GN), w = i - g * (MT * GN);
        n = g * GN + w % GN;
        m = w / GN;
    } else {
        const int w = i - in_full, gn = NT - full * GN;
        n = full * GN + w % gn;
        m = w / gn;
    }
}

// Statistics of one (row, tile) from its bf16 logits.  MODE 0: (m, s) with
// m the max logit and s = sum exp(x - m).  MODE 1: the loss's first-pass
// record of the capped, scaled logits zs = s c tanh(x / c) log2(e) (c = 0:
// s x log2(e)), base 2: (m2, S, E, X) with m2 = max zs, S = sum 2^(zs - m2),
// E = sum 2^(zs - m2) (zs - m2) and X = max |x| (which picks the loss
// kernel's tanh form).  MODE 2: MODE 1's record and, apart, the tile's sum at
// the distillation temperature T, S_T = sum 2^((zs - m2) / T).
// The statistics modes' per-logit arithmetic, one MUFU op each (relative
// error ~2^-22): the records feed the loss's normalisers, which the 16-bit
// gradient needs to ~2^-9 only.
__device__ __forceinline__ float ex2_mufu(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_mufu(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// tanh(y) = sign(y) (1 - w) / (1 + w), w = 2^(-2 log2(e) |y|) in (0, 1]
__device__ __forceinline__ float tanh_mufu(float y) {
    const float w = ex2_mufu(-2.8853900817779268f * fabsf(y));
    return copysignf((1.f - w) * rcp_mufu(1.f + w), y);
}

struct Xform {
    float c, invc, k;  // softcap (0: off), 1 / c, s * c * log2(e) (c = 0: s * log2(e))
    float invT;        // MODE 2: 1 / T
    float* st_out;     // MODE 2: N x NT sums at temperature T
};

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap map_h,
                       const __grid_constant__ CUtensorMap map_w,
                       const __grid_constant__ CUtensorMap map_o, int D, int MT, int NT,
                       void* __restrict__ stats_out, Xform xf, int* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;    // [2] accumulator written
    uint64_t* tempty = tfull + 2;        // [2] accumulator drained (one arrive per epilogue warp)
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / BK;
    const int T = MT * NT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(su32(&full[s]), 1);
            mbar_init(su32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(su32(&tfull[a]), 1);
            mbar_init(su32(&tempty[a]), EPI_WARPS);
        }
        mbar_init(su32(mma_done), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // the whole warp allocates TMEM
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            uint32_t it = 0;                 // k blocks issued, over all tiles
            uint32_t last_par[STAGES] = {};  // parity of each stage's last issued fill
            uint32_t used = 0;               // stages filled at least once
            bool go = true;
            for (int i = blockIdx.x; go && i < T; i += gridDim.x) {
                int m, n;
                tile_of(i, MT, NT, m, n);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = int(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase(su32(&empty[s]), ph ^ 1u, abort, err)) {
                        go = false;
                        break;
                    }
                    const uint32_t a = su32(smem + RING_OFF + s * STAGE_BYTES), b = a + A_BYTES;
                    mbar_expect_tx(su32(&full[s]), STAGE_BYTES);
                    tma_load_2d(a, &map_h, kb * BK, m * BM, su32(&full[s]));
                    tma_load_2d(b, &map_w, kb * BK, n * BN, su32(&full[s]));
                    last_par[s] = ph;
                    used |= 1u << s;
                }
            }
            // every fill issued has landed before shared memory is released
            for (int s = 0; s < STAGES; ++s)
                if (used & (1u << s)) drain_phase(su32(&full[s]), last_par[s], err);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = instr_desc();
            uint32_t it = 0;
            int j = 0;  // tiles of this CTA
            bool go = true, issued = false;
            for (int i = blockIdx.x; go && i < T; i += gridDim.x, ++j) {
                const int acc = j & 1;
                if (!wait_phase(su32(&tempty[acc]), (uint32_t(j >> 1) & 1u) ^ 1u, abort, err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t td = tmem + uint32_t(acc * BN);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = int(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_phase(su32(&full[s]), ph, abort, err)) {
                        go = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a = su32(smem + RING_OFF + s * STAGE_BYTES), b = a + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // 16 bf16 = 32 bytes along K per MMA
                        mma_bf16(td, smem_desc(a + 32 * k), smem_desc(b + 32 * k), idesc,
                                 (kb | k) != 0);
                    mma_commit(su32(&empty[s]));
                    issued = true;
                }
                if (go) mma_commit(su32(&tfull[acc]));
            }
            // every MMA issued has completed before TMEM is released
            if (issued) {
                mma_commit(su32(mma_done));
                drain_phase(su32(mma_done), 0u, err);
            }
        }
    } else {  // epilogue: warp w reads TMEM lane quadrant (w % 4)
        const int q = warp & 3;
        const int e = warp - 2;  // staging buffers of this warp
        unsigned char* outb = smem + OUT_OFF + e * 2 * OUT_BYTES;
        int step = 0;  // staged stores of this warp
        int j = 0;
        for (int i = blockIdx.x; i < T; i += gridDim.x, ++j) {
            int m, n;
            tile_of(i, MT, NT, m, n);
            const int acc = j & 1;
            if (!wait_phase(su32(&tfull[acc]), uint32_t(j >> 1) & 1u, abort, err)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t tbase = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc * BN);
            float mx = -INFINITY, ssum = 0.f, esum = 0.f, ax = 0.f, tsum = 0.f;
            for (int g = 0; g < BN / OUT_COLS; ++g, ++step) {
                unsigned char* ob = outb + (step & 1) * OUT_BYTES;
                // the store that last read this buffer has finished reading it
                if (lane == 0) bulk_wait_read1();
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float v[32];
                    tmem_ld32(tbase + uint32_t(g * OUT_COLS + 32 * h), v);
                    uint32_t pk[16];
                    float cm = -INFINITY;
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * t], v[2 * t + 1]);
                        pk[t] = *reinterpret_cast<const uint32_t*>(&b2);
                        v[2 * t] = __low2float(b2);
                        v[2 * t + 1] = __high2float(b2);
                        if (MODE >= 1) {  // zs of the bf16 logits, their largest |x|
                            ax = fmaxf(ax, fmaxf(fabsf(v[2 * t]), fabsf(v[2 * t + 1])));
                            v[2 * t] = xf.c > 0.f ? xf.k * tanh_mufu(v[2 * t] * xf.invc)
                                                  : xf.k * v[2 * t];
                            v[2 * t + 1] = xf.c > 0.f ? xf.k * tanh_mufu(v[2 * t + 1] * xf.invc)
                                                      : xf.k * v[2 * t + 1];
                        }
                        cm = fmaxf(cm, fmaxf(v[2 * t], v[2 * t + 1]));
                    }
                    const float nm = fmaxf(mx, cm);
                    if (MODE == 0) {
                        ssum *= exp2f((mx - nm) * 1.4426950408889634f);
#pragma unroll
                        for (int t = 0; t < 32; ++t) ssum += exp2f((v[t] - nm) * 1.4426950408889634f);
                    } else {
                        // rescale the running sums to the new max, then add the chunk
                        const float dm = mx == -INFINITY ? 0.f : mx - nm;
                        const float al = ex2_mufu(dm);
                        esum = al * (esum + dm * ssum);
                        ssum *= al;
                        if (MODE == 2) tsum *= ex2_mufu(dm * xf.invT);
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            const float d = v[t] - nm;
                            const float e = ex2_mufu(d);
                            ssum += e;
                            esum = fmaf(e, d, esum);
                            if (MODE == 2) tsum += ex2_mufu(d * xf.invT);
                        }
                    }
                    mx = nm;
                    // row `lane`, 16-byte chunks 4h .. 4h+3 of this 128-byte row,
                    // placed by the 128-byte swizzle (chunk index ^ row % 8)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = (4 * h + c) ^ (lane & 7);
                        *reinterpret_cast<uint4*>(ob + lane * 128 + chunk * 16) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                }
                // the staged rows are visible to the TMA engine, then one lane stores them
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_o, n * BN + g * OUT_COLS, m * BM + 32 * q, su32(ob));
                    bulk_commit();
                }
            }
            // this warp is done with the accumulator: the MMAs may refill it
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(su32(&tempty[acc]));
            const size_t si = size_t(m * BM + 32 * q + lane) * NT + n;
            if (MODE == 0) static_cast<float2*>(stats_out)[si] = make_float2(mx, ssum);
            else static_cast<float4*>(stats_out)[si] = make_float4(mx, ssum, esum, ax);
            if (MODE == 2) xf.st_out[si] = tsum;
        }
        if (lane == 0) bulk_wait_all();  // stores complete before shared memory is released
        __syncwarp();
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// rows x cols bf16, row-major; box = box_rows x box_cols, 128-byte swizzle
// (box_cols bf16 = 128 bytes)
int make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols) {
    auto fn = encode_fn();
    if (!fn) return 1;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 2;
}

}  // namespace hl_lmhead

namespace hl_lmhead {

int launch(int mode, const void* hidden, const void* weight, int N, int D, int V, float softcap,
           float logits_scale, void* logits, void* stats, int* err, void* stream,
           float temperature = 1.f, float* stats_t = nullptr) {
    if (N <= 0 || D <= 0 || V <= 0 || N % BM || V % BN || D % BK) return HEADLOSS_ERR_ARG;
    if (!hidden || !weight || !logits || !stats || !err) return HEADLOSS_ERR_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap) || !(logits_scale > 0.f) || !isfinite(logits_scale))
        return HEADLOSS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(weight) |
         reinterpret_cast<uintptr_t>(logits)) & 15)
        return HEADLOSS_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(stats) & (mode == 0 ? 7 : 15)) return HEADLOSS_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(err) & 3) return HEADLOSS_ERR_ALIGN;
    if (mode == 2 && (!stats_t || !(temperature > 0.f) || !isfinite(temperature)))
        return HEADLOSS_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(stats_t) & 3) return HEADLOSS_ERR_ALIGN;
    CUtensorMap mh, mw, mo;
    if (make_map(&mh, hidden, N, D, BM, BK) || make_map(&mw, weight, V, D, BN, BK) ||
        make_map(&mo, logits, N, V, 32, OUT_COLS))
        return HEADLOSS_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    const void* fn = mode == 0   ? reinterpret_cast<const void*>(&lmhead_gemm_kernel<0>)
                     : mode == 1 ? reinterpret_cast<const void*>(&lmhead_gemm_kernel<1>)
                                 : reinterpret_cast<const void*>(&lmhead_gemm_kernel<2>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    const int MT = N / BM, NT = V / BN;
    const int tiles = MT * NT;
    const int grid = tiles < sms ? tiles : sms;
    Xform xf;
    xf.c = softcap;
    xf.invc = softcap > 0.f ? 1.f / softcap : 0.f;
    xf.k = (softcap > 0.f ? logits_scale * softcap : logits_scale) * 1.4426950408889634f;
    xf.invT = 1.f / temperature;
    xf.st_out = stats_t;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (mode == 0)
        lmhead_gemm_kernel<0><<<grid, THREADS, SMEM_BYTES, s>>>(mh, mw, mo, D, MT, NT, stats, xf,
                                                                 err);
    else if (mode == 1)
        lmhead_gemm_kernel<1><<<grid, THREADS, SMEM_BYTES, s>>>(mh, mw, mo, D, MT, NT, stats, xf,
                                                                 err);
    else
        lmhead_gemm_kernel<2><<<grid, THREADS, SMEM_BYTES, s>>>(mh, mw, mo, D, MT, NT, stats, xf,
                                                                 err);
    return cudaGetLastError() == cudaSuccess ? HEADLOSS_OK : HEADLOSS_ERR_CUDA;
}

}  // namespace hl_lmhead

// The C ABI calls (include/headloss_lmhead.h documents them).
extern "C" int headloss_lmhead_logits(const void* hidden, const void* weight, int N, int D, int V,
                                      void* logits, void* stats, int* err, void* stream) {
    return hl_lmhead::launch(0, hidden, weight, N, D, V, 0.f, 1.f, logits, stats, err, stream);
}

extern "C" int headloss_lmhead_logits_rowstats(const void* hidden, const void* weight, int N,
                                               int D, int V, float softcap, float logits_scale,
                                               float temperature, void* logits, void* row_stats,
                                               float* row_stats_t, int* err, void* stream) {
    return hl_lmhead::launch(row_stats_t ? 2 : 1, hidden, weight, N, D, V, softcap, logits_scale,
                             logits, row_stats, err, stream, temperature, row_stats_t);
}
