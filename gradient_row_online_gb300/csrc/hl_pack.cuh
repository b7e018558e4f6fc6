// hl_pack.cuh -- packed-pair fp32 arithmetic (sm_100+ f32x2 instructions) and
// single-instruction MUFU wrappers for the 16-bit row kernel.
//
// A pair of fp32 values lives in one 64-bit register pair; every add / sub /
// mul / fma on a pair is one issued instruction.  All carry an explicit .rn,
// which also keeps them from being contracted.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace hl {

typedef unsigned long long f2;  // {lo, hi} fp32 pair

__device__ __forceinline__ f2 pk(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2 pk1(float v) { return pk(v, v); }
__device__ __forceinline__ void upk(f2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// 2^x, one MUFU op; results below the fp32 normal range flush to +0.
__device__ __forceinline__ float ex2f(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// log2(x), one MUFU op (approximate; x > 0 normal)
__device__ __forceinline__ float lg2f(float x) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcpf(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ f2 ex2p(f2 x) {
    float a, b;
    upk(x, a, b);
    return pk(ex2f(a), ex2f(b));
}
__device__ __forceinline__ f2 rcpp(f2 x) {
    float a, b;
    upk(x, a, b);
    return pk(rcpf(a), rcpf(b));
}
__device__ __forceinline__ float lo_of(f2 v) {
    float a, b;
    upk(v, a, b);
    return a;
}
__device__ __forceinline__ float hsum(f2 v) {
    float a, b;
    upk(v, a, b);
    return a + b;
}

// tanh(y) and 1 - tanh^2 from w = exp(-2|y|) in (0, 1], r = 1 / (1 + w):
// |tanh| = 1 - 2 w r and 1 - tanh^2 = 4 w r^2, with the sign of y put back.
// w never overflows, and 1 - tanh^2 keeps its relative accuracy where tanh
// saturates (formed as 1 - tanh^2 it would cancel) until w itself leaves
// fp32's normal range (|y| > 43).  The argument is a2x = 2 * log2(e) * y.
// One ex2 and one rcp per element; absolute tanh error ~3e-7.
struct TanhD2 {
    f2 th, omt;  // tanh, 1 - tanh^2
};
__device__ __forceinline__ TanhD2 tanh_from_ex2_arg(f2 a2x) {
    const f2 one = pk1(1.f), m2 = pk1(-2.f), four = pk1(4.f);
    float a, b;
    upk(a2x, a, b);
    const f2 w = pk(ex2f(-fabsf(a)), ex2f(-fabsf(b)));
    const f2 r = rcpp(add2(w, one));
    const f2 wr = mul2(w, r);
    float ta, tb;
    upk(fma2(wr, m2, one), ta, tb);
    TanhD2 o;
    o.th = pk(copysignf(ta, a), copysignf(tb, b));
    o.omt = mul2(wr, mul2(r, four));
    return o;
}

// ---- 16-bit storage formats: a 32-bit word holds elements (2i, 2i+1) ----

template <typename DT>
struct Pack16;

template <>
struct Pack16<__nv_bfloat16> {
    static constexpr uint32_t NEG_INF2 = 0xff80ff80u;
    __device__ static f2 unpack(uint32_t u) {
        return pk(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    __device__ static uint32_t pack(f2 g) {
        float a, b;
        upk(g, a, b);
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
        return r;
    }
    __device__ static uint32_t max2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    // magnitude max(|a|, |b|) per half (the sign bit is not meaningful)
    __device__ static uint32_t absmax2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    __device__ static float to_f(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
    __device__ static uint16_t from_f(float v) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t*>(&b);
    }
};

template <>
struct Pack16<__half> {
    static constexpr uint32_t NEG_INF2 = 0xfc00fc00u;
    __device__ static f2 unpack(uint32_t u) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u));
        return pk(f.x, f.y);
    }
    __device__ static uint32_t pack(f2 g) {
        float a, b;
        upk(g, a, b);
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
        return r;
    }
    __device__ static uint32_t max2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    // magnitude max(|a|, |b|) per half (the sign bit is not meaningful)
    __device__ static uint32_t absmax2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
    __device__ static float to_f(uint16_t h) {
        return __half2float(*reinterpret_cast<const __half*>(&h));
    }
    __device__ static uint16_t from_f(float v) {
        __half b = __float2half_rn(v);
        return *reinterpret_cast<uint16_t*>(&b);
    }
};

}  // namespace hl
