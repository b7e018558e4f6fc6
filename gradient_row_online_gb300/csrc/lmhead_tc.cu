// lmhead_tc.cu -- the LM-head GEMM in front of the loss, on the 5th-gen
// tensor cores: logits = hidden . weight^T (bf16 in, fp32 accumulation in
// TMEM, bf16 out) and, per (row, 256-column tile), the row statistics
// (max, sum of exp(x - max)) of the bf16-rounded logits.  It is the first
// building block of the fused LM head (the head GEMM whose output the loss
// consumes; tied embeddings and the LM head are PR #549 "Correctness" axes);
// the loss kernels do not call it yet.
//
// One CTA per 128 x 256 tile, 192 threads:
//   warp 0: TMA producer (one elected thread), 4-stage ring of hidden
//           128 x 64 and weight 256 x 64 bf16 tiles, 128-byte swizzle
//   warp 1: TMEM allocation (256 columns) and MMA issue (one thread),
//           tcgen05.mma kind::f16, M = 128, N = 256, K = 16, committed to the
//           stage's "empty" barrier and, after the last K block, to "acc full"
//   warps 2..5: epilogue, one TMEM lane (= one tile row) per thread
// Every wait is bounded; a wait that gives up sets *err and moves on.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "headloss.h"
#include "headloss_lmhead.h"

namespace hl_lmhead {

constexpr int BM = 128, BN = 256, BK = 64;  // BK bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;  // + alignment + barriers
constexpr long long WAIT_LIMIT = 1ll << 26;                     // polls before giving up

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
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, int* err) {
    for (long long i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try(bar, parity)) return;
    atomicOr(err, 1);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
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

__global__ void __launch_bounds__(THREADS, 1)
    lmhead_tile_kernel(const __grid_constant__ CUtensorMap map_h,
                       const __grid_constant__ CUtensorMap map_w, int D, int V,
                       __nv_bfloat16* __restrict__ logits, float2* __restrict__ stats, int* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int nk = D / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(su32(&full[s]), 1);
            mbar_init(su32(&empty[s]), 1);
        }
        mbar_init(su32(acc_full), 1);
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
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = uint32_t(kb / STAGES) & 1u;
                mbar_wait(su32(&empty[s]), ph ^ 1u, err);
                const uint32_t a = su32(smem + s * STAGE_BYTES), b = a + A_BYTES;
                mbar_expect_tx(su32(&full[s]), STAGE_BYTES);
                tma_load_2d(a, &map_h, kb * BK, m0, su32(&full[s]));
                tma_load_2d(b, &map_w, kb * BK, n0, su32(&full[s]));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t idesc = instr_desc();
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % STAGES;
                const uint32_t ph = uint32_t(kb / STAGES) & 1u;
                mbar_wait(su32(&full[s]), ph, err);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a = su32(smem + s * STAGE_BYTES), b = a + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)  // 16 bf16 = 32 bytes along K per MMA
                    mma_bf16(tmem, smem_desc(a + 32 * k), smem_desc(b + 32 * k), idesc,
                             (kb | k) != 0);
                mma_commit(su32(&empty[s]));
            }
            mma_commit(su32(acc_full));
        }
    } else {  // epilogue: warps 2..5 read TMEM lane quadrant (warp % 4)
        const int q = warp & 3;
        const int row = m0 + 32 * q + lane;
        mbar_wait(su32(acc_full), 0u, err);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        float m = -INFINITY, ssum = 0.f;
        for (int j = 0; j < BN / 32; ++j) {
            float v[32];
            tmem_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(32 * j), v);
            __nv_bfloat16 hb[32];
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                hb[i] = __float2bfloat16_rn(v[i]);
                v[i] = __bfloat162float(hb[i]);
                cm = fmaxf(cm, v[i]);
            }
            const float nm = fmaxf(m, cm);
            ssum *= exp2f((m - nm) * 1.4426950408889634f);
#pragma unroll
            for (int i = 0; i < 32; ++i) ssum += exp2f((v[i] - nm) * 1.4426950408889634f);
            m = nm;
            uint4* dst = reinterpret_cast<uint4*>(logits + size_t(row) * V + n0 + 32 * j);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = reinterpret_cast<const uint4*>(hb)[i];
        }
        stats[size_t(row) * (V / BN) + blockIdx.x] = make_float2(m, ssum);
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
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

// rows x cols bf16, row-major; box = box_rows x 64 columns, 128-byte swizzle
int make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return 1;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 2;
}

}  // namespace hl_lmhead

// The C ABI call (include/headloss_lmhead.h documents it).
extern "C" int headloss_lmhead_logits(const void* hidden, const void* weight, int N, int D, int V,
                                      void* logits, void* stats, int* err, void* stream) {
    using namespace hl_lmhead;
    if (N <= 0 || D <= 0 || V <= 0 || N % BM || V % BN || D % BK) return HEADLOSS_ERR_ARG;
    if (!hidden || !weight || !logits || !stats || !err) return HEADLOSS_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(weight) |
         reinterpret_cast<uintptr_t>(logits)) & 15)
        return HEADLOSS_ERR_ALIGN;
    CUtensorMap mh, mw;
    if (make_map(&mh, hidden, N, D, BM) || make_map(&mw, weight, V, D, BN)) return HEADLOSS_ERR_CUDA;
    if (cudaFuncSetAttribute(lmhead_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
        return HEADLOSS_ERR_CUDA;
    dim3 grid(V / BN, N / BM);
    lmhead_tile_kernel<<<grid, THREADS, SMEM_BYTES, reinterpret_cast<cudaStream_t>(stream)>>>(
        mh, mw, D, V, static_cast<__nv_bfloat16*>(logits), static_cast<float2*>(stats), err);
    return cudaGetLastError() == cudaSuccess ? HEADLOSS_OK : HEADLOSS_ERR_CUDA;
}
