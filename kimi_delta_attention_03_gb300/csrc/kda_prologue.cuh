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

}  // namespace kda
