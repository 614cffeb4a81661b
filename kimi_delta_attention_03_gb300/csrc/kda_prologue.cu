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
// HBM-bound: 1,026 bytes read and 1,026 written per row; the grid is persistent and every warp
// keeps its next row's loads in flight while it computes the current one.
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

// The raw inputs of one row, as this lane loads them.
struct ProRow {
    uint4 qk;     // eight q channels (lanes 0-15) or eight k channels (lanes 16-31)
    uint2 v, g;   // four channels each
    float b;      // beta logit (lane 0)
    float4 dt;    // dt_bias of the lane's four g channels
};

__device__ __forceinline__ ProRow load_row(const bf16* __restrict__ q_raw,
                                           const bf16* __restrict__ k_raw,
                                           const bf16* __restrict__ v_raw,
                                           const bf16* __restrict__ g_raw,
                                           const bf16* __restrict__ beta_logit,
                                           const float* __restrict__ dt_bias, int64_t row, int h,
                                           int lane) {
    ProRow r;
    const int64_t base = row * kDim;
    r.qk = __ldcs(reinterpret_cast<const uint4*>((lane < 16 ? q_raw : k_raw) + base +
                                                 8 * (lane & 15)));
    r.v = __ldcs(reinterpret_cast<const uint2*>(v_raw + base + 4 * lane));
    r.g = __ldcs(reinterpret_cast<const uint2*>(g_raw + base + 4 * lane));
    r.b = lane == 0 ? __bfloat162float(beta_logit[row]) : 0.f;
    r.dt = dt_bias ? *reinterpret_cast<const float4*>(dt_bias + h * kDim + 4 * lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    return r;
}

// Persistent grid: each warp walks rows in strides of the grid and loads its next row while it
// computes the current one, so two rows per warp are in flight.
__global__ void __launch_bounds__(kProThreads)
kda_prologue_kernel(const bf16* __restrict__ q_raw, const bf16* __restrict__ k_raw,
                    const bf16* __restrict__ v_raw, const bf16* __restrict__ g_raw,
                    const bf16* __restrict__ beta_logit, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, float lower_bound, float q_scale,
                    bf16* __restrict__ q, bf16* __restrict__ k, bf16* __restrict__ v,
                    bf16* __restrict__ g, bf16* __restrict__ beta, int64_t rows, int H) {
    // every head's gate rate, once per CTA (dynamic shared memory of H floats)
    extern __shared__ float s_na[];
    for (int i = threadIdx.x; i < H; i += kProThreads) s_na[i] = pro_gate_rate(A_log, i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kProThreads / 32);
    int64_t row = (int64_t)blockIdx.x * (kProThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    int h = (int)(row % H);
    const int h_step = (int)(warps % H);  // the head advances by this much per row step
    ProRow cur = load_row(q_raw, k_raw, v_raw, g_raw, beta_logit, dt_bias, row, h, lane);
    while (true) {
        const int64_t next = row + warps;
        const int hn = h + h_step >= H ? h + h_step - H : h + h_step;
        ProRow nxt = cur;
        if (next < rows) nxt = load_row(q_raw, k_raw, v_raw, g_raw, beta_logit, dt_bias, next, hn, lane);
        const int64_t base = row * kDim;
        const bool is_q = lane < 16;  // lanes 0-15: the q row; lanes 16-31: the k row
        {   // q or k: Swish, then the row norm
            float x[8];
            unpack8_bf16(cur.qk, x);
            pro_swish_l2_packed(x, is_q ? q_scale : 1.f);  // the packing rounds them to bf16
            __stcs(reinterpret_cast<uint4*>((is_q ? q : k) + base + 8 * (lane & 15)),
                   make_uint4(pack2_bf16(x[0], x[1]), pack2_bf16(x[2], x[3]),
                              pack2_bf16(x[4], x[5]), pack2_bf16(x[6], x[7])));
        }
        {   // v: Swish; g: the bounded gate (four channels per lane)
            const float na = s_na[h];
            const float dt[4] = {cur.dt.x, cur.dt.y, cur.dt.z, cur.dt.w};
            const uint32_t vw[2] = {cur.v.x, cur.v.y}, gw[2] = {cur.g.x, cur.g.y};
            uint32_t vo[2], go[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 vv = make_float2(__uint_as_float(vw[i] << 16),
                                              __uint_as_float(vw[i] & 0xffff0000u));
                const float2 gg = make_float2(__uint_as_float(gw[i] << 16),
                                              __uint_as_float(gw[i] & 0xffff0000u));
                const float2 hh = mul_f32x2(make_float2(0.5f, 0.5f), vv);  // Swish, in pairs
                const float2 sw = fma_f32x2(hh, make_float2(tanh_sfu(hh.x), tanh_sfu(hh.y)), hh);
                vo[i] = pack2_bf16(sw.x, sw.y);
                const float2 ga = pro_gate2_dt(gg, make_float2(dt[2 * i], dt[2 * i + 1]), na,
                                               lower_bound);
                go[i] = pack2_bf16(ga.x, ga.y);
            }
            __stcs(reinterpret_cast<uint2*>(v + base + 4 * lane), make_uint2(vo[0], vo[1]));
            __stcs(reinterpret_cast<uint2*>(g + base + 4 * lane), make_uint2(go[0], go[1]));
        }
        if (lane == 0) beta[row] = __float2bfloat16_rn(pro_sigmoid(cur.b));
        if (next >= rows) break;
        row = next;
        h = hn;
        cur = nxt;
    }
}

// ---- the short convolution in front of the prologue ----
// Causal depthwise convolution of kernel 4 along each sequence's tokens, y_t = sum_j w_j x_{t-3+j}
// per (head, channel), with the 3 inputs before a sequence's first token taken from its cache
// ("How Kimi K3 Engineered Its Way to the Frontier", section "What the hybrid saves": three
// ShortConv caches of kernel size 4 per layer).  Cache layout: bf16 [N][3 tensors q, k, v][3
// inputs, oldest first][H][128].  The convolution is in fp32 and feeds the prologue unrounded.

constexpr int kConvRun = 64;  // consecutive tokens of one head per warp

// x_{tp} of `src` for one lane's channels: a raw row of the sequence, or the cache before it
template <int kN>
__device__ __forceinline__ void conv_tap(const bf16* __restrict__ src, const bf16* __restrict__ cache,
                                         int64_t tp, int64_t a, int n, int tensor, int h, int H,
                                         int ch, float (&x)[kN]) {
    const bf16* p = nullptr;
    if (tp >= a) p = src + (tp * H + h) * kDim + ch;
    else if (cache) p = cache + ((((int64_t)n * 3 + tensor) * 3 + (tp - a + 3)) * H + h) * kDim + ch;
    if (!p) {
#pragma unroll
        for (int i = 0; i < kN; ++i) x[i] = 0.f;
        return;
    }
    if constexpr (kN == 8) {
        unpack8_bf16(*reinterpret_cast<const uint4*>(p), x);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    }
}

// The convolution along a run of tokens for one lane's kN channels of one tensor: the window
// x_{t-3} .. x_t slides one token per step (refilled from the cache or zeros at each sequence
// start); the taps are re-read each step from shared memory, where the CTA staged its head's
// taps so that each tap's four-channel vectors lie contiguous across the lanes (tp[j * kStride +
// 4 (kN / 4) h4] for tap j and channel quad h4 of this lane), and taps 0..3 accumulate in that
// order.
template <int kN>
struct ConvLane {
    const float4* tp;  // the lane's first channel quad of tap 0
    static constexpr int kStride = 32;  // float4 between taps
    float win[3][kN];  // x_{t-3}, x_{t-2}, x_{t-1}
    __device__ __forceinline__ void fill(const bf16* __restrict__ src, const bf16* __restrict__ cache,
                                         int64_t t, int64_t a, int n, int tensor, int h, int H,
                                         int ch) {
#pragma unroll
        for (int j = 0; j < 3; ++j) conv_tap<kN>(src, cache, t - 3 + j, a, n, tensor, h, H, ch, win[j]);
    }
    __device__ __forceinline__ void step(const float (&x)[kN], float (&y)[kN]) {
#pragma unroll
        for (int h4 = 0; h4 < kN / 4; ++h4) {
            float w[4][4];  // w[j][c]: tap j of channel 4 h4 + c
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 t = tp[j * kStride + 16 * h4];
                w[j][0] = t.x; w[j][1] = t.y; w[j][2] = t.z; w[j][3] = t.w;
            }
#pragma unroll
            for (int c = 0; c < 4; c += 2) {  // two channels per packed FMA, each in tap order
                const int i = 4 * h4 + c;
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    acc = fma_f32x2(make_float2(w[j][c], w[j][c + 1]),
                                    make_float2(win[j][i], win[j][i + 1]), acc);
                acc = fma_f32x2(make_float2(w[3][c], w[3][c + 1]), make_float2(x[i], x[i + 1]), acc);
                y[i] = acc.x;
                y[i + 1] = acc.y;
#pragma unroll
                for (int e = i; e < i + 2; ++e) {
                    win[0][e] = win[1][e];
                    win[1][e] = win[2][e];
                    win[2][e] = x[e];
                }
            }
        }
    }
};

// cp.async of one lane's bytes into shared memory (16, 8 or 4 bytes; both addresses aligned)
template <int kBytes>
__device__ __forceinline__ void cp_async(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "n"(kBytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// One CTA per (head, group of 8 runs of kConvRun consecutive tokens), one run per warp; runs may
// cross sequence boundaries.  The CTA stages its head's taps in shared memory once.  The raw rows
// stream through a per-warp ring of kConvStages token slots in shared memory, filled with
// cp.async kConvStages tokens ahead (each lane copies, and later reads, only its own bytes), so
// every warp keeps several rows in flight without spending registers on them.  beta takes one
// token per lane, 32 tokens at a time.
constexpr int kConvStages = 4;
struct ConvSlot {
    uint4 qk[32];  // lane l: eight q (l < 16) or k channels
    uint2 v[32];   // lane l: four v channels
    uint2 g[32];   // lane l: four g channels
};
__global__ void __launch_bounds__(kProThreads)
kda_prologue_conv_kernel(const bf16* __restrict__ q_raw, const bf16* __restrict__ k_raw,
                         const bf16* __restrict__ v_raw, const bf16* __restrict__ g_raw,
                         const bf16* __restrict__ beta_logit, const float* __restrict__ A_log,
                         const float* __restrict__ dt_bias, float lower_bound, float q_scale,
                         const float* __restrict__ w_q, const float* __restrict__ w_k,
                         const float* __restrict__ w_v, const bf16* __restrict__ cache,
                         const int32_t* __restrict__ cu_seqlens, int num_seqs,
                         bf16* __restrict__ q, bf16* __restrict__ k, bf16* __restrict__ v,
                         bf16* __restrict__ g, bf16* __restrict__ beta, int64_t T, int H) {
    __shared__ ConvSlot ring[kProThreads / 32][kConvStages];
    // the head's taps: q, k as [tensor][tap][channel half][16 lanes] float4, then v as
    // [tap][32 lanes] float4 (see ConvLane)
    __shared__ float4 taps[3 * 128];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    ConvSlot* slots = ring[warp];
    const bool is_q = lane < 16;  // lanes 0-15: q channels; lanes 16-31: k channels
    const int chqk = 8 * (lane & 15), chv = 4 * lane;
    constexpr int kWarps = kProThreads / 32;
    const int64_t runs = (T + kConvRun - 1) / kConvRun;
    const int64_t groups = (runs + kWarps - 1) / kWarps;
    int staged = -1;  // head whose taps are in shared memory
    for (int64_t citem = blockIdx.x; citem < groups * H; citem += gridDim.x) {
        const int h = (int)(citem / groups);
        const int64_t run = (citem % groups) * kWarps + warp;
        if (h != staged) {
            __syncthreads();  // every warp is done with the previous head's taps
            float* tf = reinterpret_cast<float*>(taps);
            for (int e = threadIdx.x; e < 3 * kDim; e += kProThreads) {
                const int t = e >> 7, c = e & (kDim - 1);
                const float* wsrc = t == 0 ? w_q : t == 1 ? w_k : w_v;
                const float4 w4 = *reinterpret_cast<const float4*>(wsrc + ((int64_t)h * kDim + c) * 4);
                const float wj[4] = {w4.x, w4.y, w4.z, w4.w};
                const int idx = t < 2 ? t * 128 + ((c >> 2) & 1) * 16 + (c >> 3)
                                      : 256 + (c >> 2);
#pragma unroll
                for (int j = 0; j < 4; ++j) tf[(idx + 32 * j) * 4 + (c & 3)] = wj[j];
            }
            __syncthreads();
            staged = h;
        }
        if (run >= runs) continue;
        const int64_t t0 = run * kConvRun;
        const int64_t t1 = t0 + kConvRun < T ? t0 + kConvRun : T;
        // the sequence of token t0: the last n with cu_seqlens[n] <= t0
        int lo = 0, hi = num_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_seqlens[mid] <= t0) lo = mid; else hi = mid;
        }
        int n = lo;
        int64_t a = cu_seqlens[n], b = cu_seqlens[n + 1];
        ConvLane<8> cqk;
        ConvLane<4> cv;
        cqk.tp = taps + (is_q ? 0 : 128) + (lane & 15);
        cv.tp = taps + 256 + lane;
        const bf16* src_qk = is_q ? q_raw : k_raw;
        const float na = pro_gate_rate(A_log, h);
        float dt[4] = {0.f, 0.f, 0.f, 0.f};
        if (dt_bias) {
            const float4 d4 = *reinterpret_cast<const float4*>(dt_bias + h * kDim + chv);
            dt[0] = d4.x; dt[1] = d4.y; dt[2] = d4.z; dt[3] = d4.w;
        }
        // token t's raw rows into its ring slot
        auto issue = [&](int64_t t) {
            ConvSlot& sl = slots[(t - t0) % kConvStages];
            const int64_t base = (t * H + h) * kDim;
            cp_async<16>(&sl.qk[lane], src_qk + base + chqk);
            cp_async<8>(&sl.v[lane], v_raw + base + chv);
            cp_async<8>(&sl.g[lane], g_raw + base + chv);
        };
        __syncwarp();  // the ring's previous run is read out
#pragma unroll
        for (int i = 0; i < kConvStages; ++i) {  // one commit group per ring slot, even if empty
            if (t0 + i < t1) issue(t0 + i);
            cp_async_commit();
        }
        cqk.fill(src_qk, cache, t0, a, n, is_q ? 0 : 1, h, H, chqk);
        cv.fill(v_raw, cache, t0, a, n, 2, h, H, chv);
        float bl = 0.f;  // beta logit of token t0 + 32 j + lane for the current block j
#pragma unroll 1
        for (int64_t t = t0; t < t1; ++t) {
            const int r = (int)(t - t0);
            if ((r & 31) == 0) {  // beta: one token per lane, the next 32 tokens
                const int64_t tb = t + lane;
                bl = tb < t1 ? __bfloat162float(beta_logit[tb * H + h]) : 0.f;
                if (tb < t1) beta[tb * H + h] = __float2bfloat16_rn(pro_sigmoid(bl));
            }
            cp_async_wait<kConvStages - 1>();  // token t's group has landed (for this lane)
            const ConvSlot& sl = slots[r % kConvStages];
            const uint4 cqk_raw = sl.qk[lane];
            const uint2 vr = sl.v[lane], gr = sl.g[lane];
            if (t + kConvStages < t1) issue(t + kConvStages);  // the slot is read: refill it
            cp_async_commit();
            if (t >= b) {  // a new sequence starts at t (skipping empty ones): refill the window
                do { ++n; a = cu_seqlens[n]; b = cu_seqlens[n + 1]; } while (t >= b);
                cqk.fill(src_qk, cache, t, a, n, is_q ? 0 : 1, h, H, chqk);
                cv.fill(v_raw, cache, t, a, n, 2, h, H, chv);
            }
            const int64_t base = (t * H + h) * kDim;
            float xqk[8], xv[4];
            unpack8_bf16(cqk_raw, xqk);
            xv[0] = __uint_as_float(vr.x << 16); xv[1] = __uint_as_float(vr.x & 0xffff0000u);
            xv[2] = __uint_as_float(vr.y << 16); xv[3] = __uint_as_float(vr.y & 0xffff0000u);
            float y[8], yv[4];
            cqk.step(xqk, y);
            cv.step(xv, yv);
            pro_swish_l2_packed(y, is_q ? q_scale : 1.f);  // the packing rounds them to bf16
            __stcs(reinterpret_cast<uint4*>((is_q ? q : k) + base + chqk),
                   make_uint4(pack2_bf16(y[0], y[1]), pack2_bf16(y[2], y[3]),
                              pack2_bf16(y[4], y[5]), pack2_bf16(y[6], y[7])));
            const float gv[4] = {__uint_as_float(gr.x << 16), __uint_as_float(gr.x & 0xffff0000u),
                                 __uint_as_float(gr.y << 16), __uint_as_float(gr.y & 0xffff0000u)};
            {  // v: Swish, in pairs
                const float2 h01 = mul_f32x2(make_float2(0.5f, 0.5f), make_float2(yv[0], yv[1]));
                const float2 h23 = mul_f32x2(make_float2(0.5f, 0.5f), make_float2(yv[2], yv[3]));
                const float2 s01 = fma_f32x2(h01, make_float2(tanh_sfu(h01.x), tanh_sfu(h01.y)), h01);
                const float2 s23 = fma_f32x2(h23, make_float2(tanh_sfu(h23.x), tanh_sfu(h23.y)), h23);
                __stcs(reinterpret_cast<uint2*>(v + base + chv),
                       make_uint2(pack2_bf16(s01.x, s01.y), pack2_bf16(s23.x, s23.y)));
            }
            {
                const float2 g01 = pro_gate2_dt(make_float2(gv[0], gv[1]), make_float2(dt[0], dt[1]),
                                                na, lower_bound);
                const float2 g23 = pro_gate2_dt(make_float2(gv[2], gv[3]), make_float2(dt[2], dt[3]),
                                                na, lower_bound);
                __stcs(reinterpret_cast<uint2*>(g + base + chv),
                       make_uint2(pack2_bf16(g01.x, g01.y), pack2_bf16(g23.x, g23.y)));
            }
        }
        cp_async_wait<0>();  // nothing of this run is in flight when the ring is reused
    }
}

// The cache after the call: each sequence's last 3 raw inputs (continuing from the cache before
// it when the sequence is shorter).  One thread per (sequence, tensor, head, channel); it reads
// all three values before writing, so cache_out may be cache_in.
__global__ void kda_conv_cache_kernel(const bf16* __restrict__ q_raw, const bf16* __restrict__ k_raw,
                                      const bf16* __restrict__ v_raw, const bf16* cache_in,
                                      bf16* cache_out, const int32_t* __restrict__ cu_seqlens,
                                      int num_seqs, int H) {
    const int64_t total = (int64_t)num_seqs * 3 * H * kDim;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % kDim);
        const int64_t r1 = e / kDim;
        const int h = (int)(r1 % H);
        const int64_t r2 = r1 / H;
        const int tensor = (int)(r2 % 3);
        const int n = (int)(r2 / 3);
        const int64_t a = cu_seqlens[n], b = cu_seqlens[n + 1];
        const bf16* src = tensor == 0 ? q_raw : tensor == 1 ? k_raw : v_raw;
        bf16 x[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int64_t p = b - 3 + i;
            if (p >= a) x[i] = src[(p * H + h) * kDim + c];
            else if (cache_in) x[i] = cache_in[((((int64_t)n * 3 + tensor) * 3 + (p - a + 3)) * H + h) * kDim + c];
            else x[i] = __float2bfloat16_rn(0.f);
        }
#pragma unroll
        for (int i = 0; i < 3; ++i)
            cache_out[((((int64_t)n * 3 + tensor) * 3 + i) * H + h) * kDim + c] = x[i];
    }
}

}  // namespace

cudaError_t launch_prologue(int64_t rows, int heads, const void* q_raw, const void* k_raw,
                            const void* v_raw, const void* g_raw, const void* beta_logit,
                            const float* A_log, const float* dt_bias, float lower_bound,
                            float q_scale, void* q, void* k, void* v, void* g, void* beta,
                            cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const size_t smem = (size_t)heads * sizeof(float);  // the per-head gate rates
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess && smem > 48 * 1024)
        err = cudaFuncSetAttribute(kda_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
    if (err == cudaSuccess)
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_prologue_kernel,
                                                            kProThreads, smem);
    if (err != cudaSuccess) return err;
    const int64_t per_block = kProThreads / 32;
    const int64_t need = (rows + per_block - 1) / per_block;
    const int64_t slots = (int64_t)(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(need < slots ? need : slots);
    kda_prologue_kernel<<<grid, kProThreads, smem, stream>>>(
        (const bf16*)q_raw, (const bf16*)k_raw, (const bf16*)v_raw, (const bf16*)g_raw,
        (const bf16*)beta_logit, A_log, dt_bias, lower_bound, q_scale, (bf16*)q, (bf16*)k,
        (bf16*)v, (bf16*)g, (bf16*)beta, rows, heads);
    return cudaGetLastError();
}

cudaError_t launch_prologue_conv(int64_t rows, int heads, int num_seqs, const void* q_raw,
                                 const void* k_raw, const void* v_raw, const void* g_raw,
                                 const void* beta_logit, const float* A_log, const float* dt_bias,
                                 float lower_bound, float q_scale, const float* w_q,
                                 const float* w_k, const float* w_v, const void* cache_in,
                                 void* cache_out, const int32_t* cu_seqlens, void* q, void* k,
                                 void* v, void* g, void* beta, cudaStream_t stream) {
    if (rows > 0) {
        const int64_t per_block = kProThreads / 32;
        const int64_t T = rows / heads;
        const int64_t runs = (T + kConvRun - 1) / kConvRun;
        const int64_t blocks = (runs + per_block - 1) / per_block * heads;  // (head, 8 runs)
        const unsigned grid = (unsigned)(blocks < (1LL << 30) ? blocks : (1LL << 30));
        kda_prologue_conv_kernel<<<grid, kProThreads, 0, stream>>>(
            (const bf16*)q_raw, (const bf16*)k_raw, (const bf16*)v_raw, (const bf16*)g_raw,
            (const bf16*)beta_logit, A_log, dt_bias, lower_bound, q_scale, w_q, w_k, w_v,
            (const bf16*)cache_in, cu_seqlens, num_seqs, (bf16*)q, (bf16*)k, (bf16*)v, (bf16*)g,
            (bf16*)beta, T, heads);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (cache_out) {
        const int64_t total = (int64_t)num_seqs * 3 * heads * kDim;
        const int64_t blocks = (total + 255) / 256;
        const unsigned grid = (unsigned)(blocks < (1LL << 30) ? blocks : (1LL << 30));
        kda_conv_cache_kernel<<<grid, 256, 0, stream>>>(
            (const bf16*)q_raw, (const bf16*)k_raw, (const bf16*)v_raw, (const bf16*)cache_in,
            (bf16*)cache_out, cu_seqlens, num_seqs, heads);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace kda
