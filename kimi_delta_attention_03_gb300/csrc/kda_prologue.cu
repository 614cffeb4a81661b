// kda_prologue.cu — the KDA input prologue as one elementwise pass over HBM.
//
// Raw per-token projections -> the recurrence's inputs (formulas and sources in
// kda_prologue.cuh):  q = Swish(q_raw) q_scale / |Swish(q_raw)|,  k = Swish(k_raw) / |Swish(k_raw)|,
// v = Swish(v_raw),  log_alpha = lb sigmoid(exp(A_log[h]) (g_raw + dt_bias[h])),
// beta = sigmoid(beta_logit).  All bf16 in and out.
//
// One warp per (token, head) row: lanes 0-15 hold the q row and lanes 16-31 the k row, eight
// consecutive channels each (one 16-byte load), the layout of the fused prefill's factor pass, so
// both reduce the row norms in the same order; v and g are four channels per lane.  The pass is
// HBM-bound: 1,026 bytes read and 1,026 written per row.
#include "kda_common.cuh"
#include "kda_prologue.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kProThreads = 256;  // 8 rows per block

__device__ __forceinline__ void unpack8_bf16(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

__global__ void __launch_bounds__(kProThreads)
kda_prologue_kernel(const bf16* __restrict__ q_raw, const bf16* __restrict__ k_raw,
                    const bf16* __restrict__ v_raw, const bf16* __restrict__ g_raw,
                    const bf16* __restrict__ beta_logit, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, float lower_bound, float q_scale,
                    bf16* __restrict__ q, bf16* __restrict__ k, bf16* __restrict__ v,
                    bf16* __restrict__ g, bf16* __restrict__ beta, int64_t rows, int H) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kProThreads / 32);
    for (int64_t row = (int64_t)blockIdx.x * (kProThreads / 32) + (threadIdx.x >> 5); row < rows;
         row += warps) {
        const int h = (int)(row % H);
        const int64_t base = row * kDim;
        // every load of the row first: one memory round trip per row
        const bool is_q = lane < 16;  // lanes 0-15: the q row; lanes 16-31: the k row
        const int64_t eqk = base + 8 * (lane & 15);
        const int64_t evg = base + 4 * lane;    // v and g: four channels per lane
        const uint4 qk = __ldcs(reinterpret_cast<const uint4*>((is_q ? q_raw : k_raw) + eqk));
        const uint2 vr = __ldcs(reinterpret_cast<const uint2*>(v_raw + evg));
        const uint2 gr = __ldcs(reinterpret_cast<const uint2*>(g_raw + evg));
        const float b_logit = lane == 0 ? __bfloat162float(beta_logit[row]) : 0.f;
        float dt[4] = {0.f, 0.f, 0.f, 0.f};
        if (dt_bias) {
            const float4 d4 = *reinterpret_cast<const float4*>(dt_bias + h * kDim + 4 * lane);
            dt[0] = d4.x; dt[1] = d4.y; dt[2] = d4.z; dt[3] = d4.w;
        }
        const float na = pro_gate_rate(A_log, h);
        {   // q or k: Swish, then the row norm
            float x[8];
            unpack8_bf16(qk, x);
            pro_swish_l2(x, is_q ? q_scale : 1.f);
            __stcs(reinterpret_cast<uint4*>((is_q ? q : k) + eqk),
                   make_uint4(pack2_bf16(x[0], x[1]), pack2_bf16(x[2], x[3]),
                              pack2_bf16(x[4], x[5]), pack2_bf16(x[6], x[7])));
        }
        {   // v: Swish; g: the bounded gate
            const uint32_t vw[2] = {vr.x, vr.y}, gw[2] = {gr.x, gr.y};
            uint32_t vo[2], go[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float v0 = __uint_as_float(vw[i] << 16), v1 = __uint_as_float(vw[i] & 0xffff0000u);
                const float g0 = __uint_as_float(gw[i] << 16), g1 = __uint_as_float(gw[i] & 0xffff0000u);
                vo[i] = pack2_bf16(pro_swish(v0), pro_swish(v1));
                go[i] = pack2_bf16(pro_gate(g0, dt[2 * i], na, lower_bound),
                                   pro_gate(g1, dt[2 * i + 1], na, lower_bound));
            }
            __stcs(reinterpret_cast<uint2*>(v + evg), make_uint2(vo[0], vo[1]));
            __stcs(reinterpret_cast<uint2*>(g + evg), make_uint2(go[0], go[1]));
        }
        if (lane == 0) beta[row] = __float2bfloat16_rn(pro_sigmoid(b_logit));
    }
}

}  // namespace

cudaError_t launch_prologue(int64_t rows, int heads, const void* q_raw, const void* k_raw,
                            const void* v_raw, const void* g_raw, const void* beta_logit,
                            const float* A_log, const float* dt_bias, float lower_bound,
                            float q_scale, void* q, void* k, void* v, void* g, void* beta,
                            cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int64_t per_block = kProThreads / 32;
    const int64_t blocks = (rows + per_block - 1) / per_block;
    const unsigned grid = (unsigned)(blocks < (1LL << 30) ? blocks : (1LL << 30));
    kda_prologue_kernel<<<grid, kProThreads, 0, stream>>>(
        (const bf16*)q_raw, (const bf16*)k_raw, (const bf16*)v_raw, (const bf16*)g_raw,
        (const bf16*)beta_logit, A_log, dt_bias, lower_bound, q_scale, (bf16*)q, (bf16*)k,
        (bf16*)v, (bf16*)g, (bf16*)beta, rows, heads);
    return cudaGetLastError();
}

}  // namespace kda
