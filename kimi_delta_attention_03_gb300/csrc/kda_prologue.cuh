// kda_prologue.cuh — elementwise arithmetic of the KDA input prologue, shared by the fused
// prefill variant and the standalone prologue kernel so that both produce the same bits.
//
// The prologue ("Kimi K3" (ai.thesatyajit.com), section "Kimi Delta Attention: constant-size
// memory over a million tokens": Swish, then L2 normalisation, for queries and keys; Swish for
// values.  "How Kimi K3 Engineered Its Way to the Frontier", section "How KDA updates its
// state": the decay gate lower_bound * sigmoid(exp(A_log) * (g + dt_bias)).  FlashKDA's forward,
// section "FlashKDA: the equation, shipped as a kernel": beta = sigmoid(beta logits)).
//
// The gate and beta use sigmoid(x) = 1 / (1 + 2^{-x log2 e}) on the SFU's exp2 and reciprocal
// approximations: about 1e-6 relative error for every x, including the small decays near 0 that
// a tanh-based form (0.5 + 0.5 tanh(x / 2)) would lose to a cancellation.  Swish uses that
// tanh form, one SFU operation instead of two: its absolute error (about |x| 2.5e-4) is small
// against the row it belongs to.  Every prologue output is rounded to bf16 where an unfused
// pipeline would store it.
#pragma once

#include <cuda_bf16.h>

#include "kda_common.cuh"

namespace kda {

constexpr float kProNormEps = 1e-6f;  // added to the sum of squares of the L2 norm

__device__ __forceinline__ float ex2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float tanh_sfu(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_sfu(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// sigmoid(x), fp32 (0 for x -> -inf, 1 for x -> +inf)
__device__ __forceinline__ float pro_sigmoid(float x) {
    return rcp_sfu(__fadd_rn(1.f, ex2_sfu(__fmul_rn(-1.4426950408889634f, x))));
}

// Swish(x) = x sigmoid(x) = h + h tanh(h) with h = x / 2
__device__ __forceinline__ float pro_swish(float x) {
    const float h = __fmul_rn(0.5f, x);
    return fmaf(h, tanh_sfu(h), h);
}

// log alpha = lb sigmoid(a (g + dt)) = lb / (1 + 2^{na (g + dt)}) with na = -a log2 e, rounded
// to bf16
__device__ __forceinline__ float pro_gate(float g, float dt, float na, float lb) {
    return round_bf16(__fmul_rn(lb, rcp_sfu(__fadd_rn(1.f, ex2_sfu(__fmul_rn(na, __fadd_rn(g, dt)))))));
}

// pro_gate of two values as packed fp32 pairs (the same operations per value, the same bits)
__device__ __forceinline__ float2 pro_gate2_dt(float2 g, float2 dt, float na, float lb) {
    const float2 y = mul_f32x2(make_float2(na, na), add_f32x2(g, dt));
    const float2 d = add_f32x2(make_float2(1.f, 1.f), make_float2(ex2_sfu(y.x), ex2_sfu(y.y)));
    const float2 z = mul_f32x2(make_float2(lb, lb), make_float2(rcp_sfu(d.x), rcp_sfu(d.y)));
    return make_float2(round_bf16(z.x), round_bf16(z.y));
}
__device__ __forceinline__ float2 pro_gate2(float2 g, float dt, float na, float lb) {
    const float2 y = mul_f32x2(make_float2(na, na), add_f32x2(g, make_float2(dt, dt)));
    const float2 d = add_f32x2(make_float2(1.f, 1.f), make_float2(ex2_sfu(y.x), ex2_sfu(y.y)));
    const float2 z = mul_f32x2(make_float2(lb, lb), make_float2(rcp_sfu(d.x), rcp_sfu(d.y)));
    return make_float2(round_bf16(z.x), round_bf16(z.y));
}

// na = -exp(A_log[h]) log2 e for head h
__device__ __forceinline__ float pro_gate_rate(const float* A_log, int h) {
    return __fmul_rn(-1.4426950408889634f, expf(A_log[h]));
}

// Sum over a 128-channel row held as eight consecutive channels per lane of a 16-lane group
// (lane & 15 = channel group): eight in-order FMAs, then a pairwise butterfly over the group.
// Every lane of the group ends with the same bits.
__device__ __forceinline__ float row_sum_squares16(const float (&x)[8]) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s = fmaf(x[j], x[j], s);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// In place: x <- round_bf16(Swish(x) * scale / sqrt(sum Swish(x)^2 + eps)) for one 128-channel
// row spread over a 16-lane group (all 32 lanes of the warp must call it together)
__device__ __forceinline__ void pro_swish_l2(float (&x)[8], float scale) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = pro_swish(x[j]);
    const float inv = __fmul_rn(rsqrtf(__fadd_rn(row_sum_squares16(x), kProNormEps)), scale);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = round_bf16(__fmul_rn(x[j], inv));
}

// pro_swish_l2 for a row of k and a row of q held by the same 16-lane group, as packed fp32
// pairs (k, q): the same operations in the same order per value, so the same bits.  The results
// are left unrounded for a caller that packs them to bf16 (which rounds them as round_bf16 would).
__device__ __forceinline__ void pro_swish_l2_kq(float (&k)[8], float (&q)[8], float q_scale) {
    float2 ss = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 hh = mul_f32x2(make_float2(0.5f, 0.5f), make_float2(k[j], q[j]));
        const float2 sw = fma_f32x2(hh, make_float2(tanh_sfu(hh.x), tanh_sfu(hh.y)), hh);
        k[j] = sw.x;
        q[j] = sw.y;
        ss = fma_f32x2(sw, sw, ss);
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, ss.x, off),
                                     __shfl_xor_sync(0xffffffffu, ss.y, off));
        ss = make_float2(__fadd_rn(ss.x, o.x), __fadd_rn(ss.y, o.y));
    }
    const float2 inv = make_float2(rsqrtf(__fadd_rn(ss.x, kProNormEps)),
                                   __fmul_rn(rsqrtf(__fadd_rn(ss.y, kProNormEps)), q_scale));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 x = mul_f32x2(make_float2(k[j], q[j]), inv);
        k[j] = x.x;
        q[j] = x.y;
    }
}

// Swish of eight values as packed fp32 pairs (the same bits as pro_swish on each)
__device__ __forceinline__ void pro_swish8(float (&x)[8]) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const float2 hh = mul_f32x2(make_float2(0.5f, 0.5f), make_float2(x[j], x[j + 1]));
        const float2 sw = fma_f32x2(hh, make_float2(tanh_sfu(hh.x), tanh_sfu(hh.y)), hh);
        x[j] = sw.x;
        x[j + 1] = sw.y;
    }
}

// pro_swish_l2 with its Swish and scaling on packed fp32 pairs, for a caller that packs the
// results to bf16 (the packing rounds them as round_bf16 would): the same bits.
__device__ __forceinline__ void pro_swish_l2_packed(float (&x)[8], float scale) {
    pro_swish8(x);
    const float inv = __fmul_rn(rsqrtf(__fadd_rn(row_sum_squares16(x), kProNormEps)), scale);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const float2 y = mul_f32x2(make_float2(x[j], x[j + 1]), make_float2(inv, inv));
        x[j] = y.x;
        x[j + 1] = y.y;
    }
}


}  // namespace kda
