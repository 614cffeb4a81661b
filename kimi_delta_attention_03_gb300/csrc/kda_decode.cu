// kda_decode.cu — single-token KDA decode: in-place state update, one pass over HBM.
//
// For one (sequence, head) unit with state S (128 x 128 fp32, row = key channel) and one
// token (q, k, v, g = log alpha, beta):
//     S <- Diag(exp(g)) S;   u = beta (v - S^T k);   S <- S + k u^T;   o = S^T q
// ("How Kimi K3 Engineered Its Way to the Frontier", section "How KDA updates its state";
// in-place update at every decoding step: "k3_training_and_infra_notes", section 4.5).
//
// The step is bound by HBM: 64 KiB of state read and 64 KiB written per unit against about
// 1.3 KFLOP per KiB.  Each CTA (256 threads) owns one unit and keeps the whole decayed state
// in registers between the read and the write, so S crosses HBM exactly twice:
//   thread (warp w, lane l) holds rows {16 w + r : r < 16}, columns 4l .. 4l+3 (one float4
//   per row; a warp touches one full 512-byte row per access, fully coalesced; its rows are
//   contiguous, so their decay, k and q scalars come four to a shared-memory load).
// The two column reductions x = (D S)^T k and y = (D S)^T q are per-thread partial sums over
// its 16 rows, then a cross-warp sum through shared memory.  The output uses the identity
//     o = S_new^T q = y + (k . q) u,
// so the updated state never has to be re-read.  Loads and stores are streaming (evict-first)
// because every byte is touched once.
#include "kda_common.cuh"
#include "kda_prologue.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;


// The input prologue of the decode variants that take raw projections (kPro): per head rate and
// bias of the gate, its lower bound, and the q scale (arithmetic in kda_prologue.cuh).
struct DecPro {
    const float* A_log;    // [H]
    const float* dt_bias;  // [H][128] or null
    float lb;
    float q_scale;
    int H;
};

// Raw projections of one token for warp_prologue.  Lane l of the warp that produces channels
// [32 cw, 32 cw + 32) holds the eight channels 8 (l & 15) .. 8 (l & 15) + 7 of k (l < 16) or q
// (l >= 16), as one 16-byte vector, and its own channel 32 cw + l of k, q, g and v.
struct RawTok {
    uint4 grp;
    __nv_bfloat16 kc, qc, gc, vc;
};

__device__ __forceinline__ void load_raw(RawTok& r, const __nv_bfloat16* k,
                                         const __nv_bfloat16* q, const __nv_bfloat16* g,
                                         const __nv_bfloat16* v, int64_t row, int cw, int lane) {
    r.grp = *reinterpret_cast<const uint4*>((lane < 16 ? k : q) + row * kDim + 8 * (lane & 15));
    const int64_t e = row * kDim + 32 * cw + lane;
    r.kc = k[e];
    r.qc = q[e];
    r.gc = g[e];
    r.vc = v[e];
}

// The prologue of one token's channels [32 cw, 32 cw + 32) by one warp, with no barrier: the
// warp forms both row norms itself and writes its channels of k and q (Swish, scaled, rounded to
// bf16), alpha = exp(gate) and v = Swish(v) (rounded to bf16).  The norms are the standalone
// prologue's: eight in-order FMAs per lane of a 16-lane group, then the sum over the group that
// its 1-2-4-8 butterfly forms, which is the balanced binary tree over the 16 lane partials (each
// pairwise addition is commutative, so every lane of the butterfly ends with exactly that tree).
// Here each lane reads its group's 16 partials from the warp's 32-float scratch in shared memory
// and adds the tree itself; two independent shuffles then hand every lane both scales.
__device__ __forceinline__ float tree_sum16(const float* p) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4),
                 c = *reinterpret_cast<const float4*>(p + 8), d = *reinterpret_cast<const float4*>(p + 12);
    const float l1[8] = {__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w), __fadd_rn(b.x, b.y),
                         __fadd_rn(b.z, b.w), __fadd_rn(c.x, c.y), __fadd_rn(c.z, c.w),
                         __fadd_rn(d.x, d.y), __fadd_rn(d.z, d.w)};
    const float l2[4] = {__fadd_rn(l1[0], l1[1]), __fadd_rn(l1[2], l1[3]), __fadd_rn(l1[4], l1[5]),
                         __fadd_rn(l1[6], l1[7])};
    return __fadd_rn(__fadd_rn(l2[0], l2[1]), __fadd_rn(l2[2], l2[3]));
}
__device__ __forceinline__ void warp_prologue(const RawTok& r, float dt, float na, float lb,
                                              float q_scale, int c, int lane, float* scratch,
                                              float* s_k, float* s_q, float* s_a, float* s_v) {
    float ss = 0.f;
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&r.grp);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(p2[j]);
        const float x0 = pro_swish(f.x), x1 = pro_swish(f.y);
        ss = fmaf(x0, x0, ss);
        ss = fmaf(x1, x1, ss);
    }
    scratch[lane] = ss;
    __syncwarp();
    const float inv = __fmul_rn(rsqrtf(__fadd_rn(tree_sum16(scratch + (lane & 16)), kProNormEps)),
                                lane < 16 ? 1.f : q_scale);
    __syncwarp();  // the scratch is rewritten by the warp's next token
    const float ik = __shfl_sync(0xffffffffu, inv, 0);
    const float iq = __shfl_sync(0xffffffffu, inv, 16);
    s_k[c] = round_bf16(__fmul_rn(pro_swish(__bfloat162float(r.kc)), ik));
    s_q[c] = round_bf16(__fmul_rn(pro_swish(__bfloat162float(r.qc)), iq));
    s_a[c] = expf(pro_gate(__bfloat162float(r.gc), dt, na, lb));
    s_v[c] = round_bf16(pro_swish(__bfloat162float(r.vc)));
}

template <typename TIn, bool kPro>
__global__ void __launch_bounds__(kDecodeThreads, 2)
kda_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                  const TIn* __restrict__ v, const TIn* __restrict__ g,
                  const TIn* __restrict__ beta, float* __restrict__ state,
                  TIn* __restrict__ out, int64_t units, const DecPro pro) {
    __shared__ __align__(16) float s_k[kDim], s_q[kDim], s_a[kDim], s_v[kDim], s_u[kDim];
    __shared__ __align__(16) float s_norm[kPro ? 4 : 1][32];  // per prologue warp: norm partials
    __shared__ __align__(16) float s_rx[8][kDim];
    __shared__ __align__(16) float s_ry[8][kDim];
    __shared__ float s_kq;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        float* S = state + unit * (int64_t)(kDim * kDim);
        float4 s[16];
        float b;
        if constexpr (kPro) {  // raw projections: the prologue first
            // The token's raw inputs are requested before the state, so that they arrive first
            // and the prologue's arithmetic (warps 0-3, 32 channels each) overlaps the state
            // stream.
            const int h = (int)(unit % pro.H);
            RawTok raw{};
            float dt = 0.f;
            if (warp < 4) {
                load_raw(raw, k, q, g, v, unit, warp, lane);
                dt = pro.dt_bias ? pro.dt_bias[h * kDim + tid] : 0.f;
            }
            const TIn rb = beta[unit];
            const float na = pro_gate_rate(pro.A_log, h);
#pragma unroll
            for (int r = 0; r < 16; ++r)
                s[r] = __ldcs(reinterpret_cast<const float4*>(S + (16 * warp + r) * kDim) + lane);
            if (warp < 4)
                warp_prologue(raw, dt, na, pro.lb, pro.q_scale, tid, lane, s_norm[warp], s_k, s_q,
                              s_a, s_v);
            b = round_bf16(pro_sigmoid(io<TIn>::to_f(rb)));
            __syncthreads();
        } else {
#pragma unroll
            for (int r = 0; r < 16; ++r)
                s[r] = __ldcs(reinterpret_cast<const float4*>(S + (16 * warp + r) * kDim) + lane);
            if (tid < kDim) {
                const int64_t e = unit * kDim + tid;
                s_k[tid] = io<TIn>::to_f(k[e]);
                s_q[tid] = io<TIn>::to_f(q[e]);
                s_a[tid] = expf(io<TIn>::to_f(g[e]));
                s_v[tid] = io<TIn>::to_f(v[e]);
            }
            b = io<TIn>::to_f(beta[unit]);
            __syncthreads();
        }

        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
        float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
#pragma unroll
        for (int r4 = 0; r4 < 16; r4 += 4) {  // the warp's rows are contiguous: four scalars a load
            const float4 a4 = *reinterpret_cast<const float4*>(s_a + 16 * warp + r4);
            const float4 k4 = *reinterpret_cast<const float4*>(s_k + 16 * warp + r4);
            const float4 q4 = *reinterpret_cast<const float4*>(s_q + 16 * warp + r4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w},
                        qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int r = r4 + m;
                const float a = av[m], kk = kv[m], qq = qv[m];
                s[r].x *= a; s[r].y *= a; s[r].z *= a; s[r].w *= a;
                x0 = fmaf(kk, s[r].x, x0); x1 = fmaf(kk, s[r].y, x1);
                x2 = fmaf(kk, s[r].z, x2); x3 = fmaf(kk, s[r].w, x3);
                y0 = fmaf(qq, s[r].x, y0); y1 = fmaf(qq, s[r].y, y1);
                y2 = fmaf(qq, s[r].z, y2); y3 = fmaf(qq, s[r].w, y3);
            }
        }
        reinterpret_cast<float4*>(s_rx[warp])[lane] = make_float4(x0, x1, x2, x3);
        reinterpret_cast<float4*>(s_ry[warp])[lane] = make_float4(y0, y1, y2, y3);
        if (warp == 0) {
            float p = 0.f;
#pragma unroll
            for (int m = 0; m < kDim / 32; ++m) p = fmaf(s_k[lane + 32 * m], s_q[lane + 32 * m], p);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (lane == 0) s_kq = p;
        }
        __syncthreads();

        if (tid < kDim) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) { x += s_rx[w][tid]; y += s_ry[w][tid]; }
            const float u = b * (s_v[tid] - x);
            s_u[tid] = u;
            out[unit * kDim + tid] = io<TIn>::from_f(fmaf(s_kq, u, y));
        }
        __syncthreads();

        const float4 u4 = reinterpret_cast<const float4*>(s_u)[lane];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float kk = s_k[16 * warp + r];
            float4 o;
            o.x = fmaf(kk, u4.x, s[r].x); o.y = fmaf(kk, u4.y, s[r].y);
            o.z = fmaf(kk, u4.z, s[r].z); o.w = fmaf(kk, u4.w, s[r].w);
            __stcs(reinterpret_cast<float4*>(S + (16 * warp + r) * kDim) + lane, o);
        }
        __syncthreads();  // shared vectors are rewritten by the next unit of this CTA
    }
}

// A run of tokens per (sequence, head) in one pass over the state: the replayed accepted
// tokens, the bonus token and the next draft window of speculative decoding share one
// recurrent loop, the state read once and written once ("k3_training_and_infra_notes",
// section 4.5, KDA decoding: cache the draft tokens' projected inputs, rebuild the accepted
// states on-chip, write back once).  Sequence n's tokens are rows cu[n] .. cu[n+1] - 1 of the
// inputs (layout [T, H, 128], as the prefill's); every token's output is written (when out is
// given) from the state after the run's earlier tokens; the state after the first commit[n]
// tokens is written back (nothing when commit[n] = 0; all of them when commit is null).  Per
// token the arithmetic is the single-token step's, in the same order.  The state is read from
// state_in (zeros when null) and written to state_out (skipped when null); the two may be the
// same array, as each unit reads its state before writing it.  A unit with no tokens copies
// its state across when the two differ.  With fp32 inputs the prefill runs through this
// kernel too: whole sequences, every token committed, exact fp32 arithmetic.
template <typename TIn, bool kPro>
__global__ void __launch_bounds__(kDecodeThreads, 2)
kda_decode_window_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                         const TIn* __restrict__ v, const TIn* __restrict__ g,
                         const TIn* __restrict__ beta, const int32_t* __restrict__ cu_seqlens,
                         const float* state_in, float* state_out, TIn* __restrict__ out,
                         const int32_t* __restrict__ commit, int64_t units, int H,
                         int64_t total_tokens, int max_len, int* status, const DecPro pro) {
    // With raw projections the prologue runs one token ahead of the recurrence, on warps 4-7
    // while warps 0-3 form the token's u, so the token vectors are double-buffered (token t in
    // buffer t & 1).
    constexpr int NB = kPro ? 2 : 1;
    __shared__ __align__(16) float s_k[NB][kDim], s_q[NB][kDim], s_a[NB][kDim], s_v[NB][kDim];
    __shared__ __align__(16) float s_u[kDim];
    __shared__ float s_b[NB];
    __shared__ __align__(16) float s_norm[kPro ? 4 : 1][32];  // per prologue warp: norm partials
    __shared__ __align__(16) float s_rx[8][kDim];
    __shared__ __align__(16) float s_ry[8][kDim];
    __shared__ float s_kq;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int64_t n = unit / H;
        const int h = (int)(unit - n * H);
        const int64_t t0 = cu_seqlens[n];
        const int64_t len64 = cu_seqlens[n + 1] - t0;
        if (t0 < 0 || len64 < 0 || t0 + len64 > total_tokens || len64 > max_len) {
            // the device cu_seqlens disagree with the host lengths the call was checked against
            if (tid == 0) report_status(status, KDA_ERR_INVALID_ARG);
            continue;
        }
        const int len = (int)len64;
        const int ncommit = commit ? min(max(commit[n], 0), len) : len;
        const float* Sin = state_in ? state_in + unit * (int64_t)(kDim * kDim) : nullptr;
        float* S = state_out ? state_out + unit * (int64_t)(kDim * kDim) : nullptr;
        if (len <= 0) {
            if (S && S != Sin)
                for (int e = tid; e < kDim * kDim / 4; e += kDecodeThreads)
                    reinterpret_cast<float4*>(S)[e] =
                        Sin ? reinterpret_cast<const float4*>(Sin)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        float4 s[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            s[r] = Sin ? __ldcs(reinterpret_cast<const float4*>(Sin + (16 * warp + r) * kDim) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        float pro_dt = 0.f, pro_na = 0.f;
        if constexpr (kPro) {  // warps 4-7 run the prologue, channel tid - 128 each
            pro_dt = pro.dt_bias && tid >= kDim ? pro.dt_bias[h * kDim + tid - kDim] : 0.f;
            pro_na = pro_gate_rate(pro.A_log, h);
        }

        // The grid is persistent: the state and the token rows of this CTA's next unit are
        // pulled into L2 while this unit's tokens run, so its loads find them there.
        const int64_t nu = unit + gridDim.x;
        if (nu < units) {
            if (tid < 4 && state_in) {
                const float* nxt = state_in + nu * (int64_t)(kDim * kDim) + tid * 4096;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], 16384;" ::"l"(nxt) : "memory");
            }
            constexpr int kLine = 128 / (int)sizeof(TIn);  // elements per 128-byte line
            constexpr int kLines = kDim / kLine;
            const int64_t nn = nu / H;
            const int nh = (int)(nu - nn * H);
            const int64_t nt0 = cu_seqlens[nn];
            const int nlen = min((int)(cu_seqlens[nn + 1] - nt0), 64);  // the first tokens
            for (int i = tid; i < nlen * 4 * kLines; i += kDecodeThreads) {
                const int tok = i / (4 * kLines), rem = i - tok * 4 * kLines;
                const int which = rem / kLines, line = rem - which * kLines;
                const TIn* src = which == 0 ? k : which == 1 ? q : which == 2 ? g : v;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(
                    src + ((nt0 + tok) * H + nh) * kDim + line * kLine));
            }
            if (tid < nlen) asm volatile("prefetch.global.L2 [%0];" ::"l"(beta + (nt0 + tid) * H + nh));
        }

        // the next token's inputs are fetched into registers while this token is computed (with
        // raw projections, by warps 4-7, two tokens ahead of the recurrence)
        TIn nk{}, nq{}, ng{}, nv{}, nb{};
        [[maybe_unused]] RawTok raw{};
        auto fetch = [&](int t) {
            const int64_t row = (t0 + t) * H + h;
            if constexpr (kPro) {
                if (tid >= kDim) {
                    load_raw(raw, k, q, g, v, row, warp - 4, lane);
                    nb = beta[row];
                }
            } else {
                if (tid < kDim) {
                    const int64_t e = row * kDim + tid;
                    nk = k[e]; nq = q[e]; ng = g[e]; nv = v[e];
                }
                nb = beta[row];
            }
        };
        // Raw projections: the fetched token's prologue into buffer `buf`, on warps 4-7.
        [[maybe_unused]] auto pro_token = [&](int buf) {
            if (tid >= kDim) {
                warp_prologue(raw, pro_dt, pro_na, pro.lb, pro.q_scale, tid - kDim, lane,
                              s_norm[warp - 4],
                              s_k[buf], s_q[buf], s_a[buf], s_v[buf]);
                if (tid == kDim) s_b[buf] = round_bf16(pro_sigmoid(io<TIn>::to_f(nb)));
            }
        };
        fetch(0);
        if constexpr (kPro) {  // token 0's prologue; later tokens' run one token ahead
            pro_token(0);
            if (1 < len) fetch(1);
            __syncthreads();
        }
#pragma unroll 1
        for (int t = 0; t < len; ++t) {
            const int64_t row = (t0 + t) * H + h;
            const int cur = kPro ? (t & 1) : 0;
            float b;
            if constexpr (kPro) {
                b = s_b[cur];
            } else {
                if (tid < kDim) {
                    s_k[0][tid] = io<TIn>::to_f(nk);
                    s_q[0][tid] = io<TIn>::to_f(nq);
                    s_a[0][tid] = expf(io<TIn>::to_f(ng));
                    s_v[0][tid] = io<TIn>::to_f(nv);
                }
                b = io<TIn>::to_f(nb);
                if (t + 1 < len) fetch(t + 1);
                __syncthreads();
            }

            float2 x01 = make_float2(0.f, 0.f), x23 = x01, y01 = x01, y23 = x01;
#pragma unroll
            for (int r4 = 0; r4 < 16; r4 += 4) {
                // contiguous rows: four scalars a load (one at a time with raw projections, whose
                // prologue already holds the registers the wider loads need)
                float av[4], kv[4], qv[4];
                if constexpr (kPro) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        av[m] = s_a[cur][16 * warp + r4 + m];
                        kv[m] = s_k[cur][16 * warp + r4 + m];
                        qv[m] = s_q[cur][16 * warp + r4 + m];
                    }
                } else {
                    const float4 a4 = *reinterpret_cast<const float4*>(&s_a[cur][16 * warp + r4]);
                    const float4 k4 = *reinterpret_cast<const float4*>(&s_k[cur][16 * warp + r4]);
                    const float4 q4 = *reinterpret_cast<const float4*>(&s_q[cur][16 * warp + r4]);
                    av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
                    kv[0] = k4.x; kv[1] = k4.y; kv[2] = k4.z; kv[3] = k4.w;
                    qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int r = r4 + m;
                    const float2 a2 = make_float2(av[m], av[m]), k2 = make_float2(kv[m], kv[m]),
                                 q2 = make_float2(qv[m], qv[m]);
                    const float2 s01 = mul_f32x2(make_float2(s[r].x, s[r].y), a2);
                    const float2 s23 = mul_f32x2(make_float2(s[r].z, s[r].w), a2);
                    s[r] = make_float4(s01.x, s01.y, s23.x, s23.y);
                    x01 = fma_f32x2(k2, s01, x01); x23 = fma_f32x2(k2, s23, x23);
                    y01 = fma_f32x2(q2, s01, y01); y23 = fma_f32x2(q2, s23, y23);
                }
            }
            reinterpret_cast<float4*>(s_rx[warp])[lane] = make_float4(x01.x, x01.y, x23.x, x23.y);
            reinterpret_cast<float4*>(s_ry[warp])[lane] = make_float4(y01.x, y01.y, y23.x, y23.y);
            if (warp == 0) {
                float p = 0.f;
#pragma unroll
                for (int m = 0; m < kDim / 32; ++m)
                    p = fmaf(s_k[cur][lane + 32 * m], s_q[cur][lane + 32 * m], p);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if (lane == 0) s_kq = p;
            }
            __syncthreads();

            [[maybe_unused]] float y_keep = 0.f;
            if constexpr (kPro) {
                if (tid < kDim) {
                    float x = 0.f, y = 0.f;
#pragma unroll
                    for (int w8 = 0; w8 < 8; ++w8) { x += s_rx[w8][tid]; y += s_ry[w8][tid]; }
                    const float u = b * (s_v[cur][tid] - x);
                    s_u[tid] = u;
                    if (out) out[row * kDim + tid] = io<TIn>::from_f(fmaf(s_kq, u, y));
                }
                // meanwhile the next token's prologue on warps 4-7, into the other buffer
                if (t + 1 < len) {
                    pro_token(cur ^ 1);
                    if (t + 2 < len) fetch(t + 2);
                }
            } else {
                // x on threads 0-127 (then u), y on threads 128-255; the output, which needs u,
                // is written in the next phase
                const int j = tid & (kDim - 1);
                const float(*part)[kDim] = tid < kDim ? s_rx : s_ry;
                float acc = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) acc += part[w8][j];
                if (tid < kDim)
                    s_u[j] = b * (s_v[cur][j] - acc);
                else
                    y_keep = acc;
            }
            __syncthreads();
            if constexpr (!kPro) {
                if (tid >= kDim && out) {
                    const int j = tid - kDim;
                    out[row * kDim + j] = io<TIn>::from_f(fmaf(s_kq, s_u[j], y_keep));
                }
            }

            const float4 u4 = reinterpret_cast<const float4*>(s_u)[lane];
            const float2 u01 = make_float2(u4.x, u4.y), u23 = make_float2(u4.z, u4.w);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float kk = s_k[cur][16 * warp + r];
                const float2 k2 = make_float2(kk, kk);
                const float2 s01 = fma_f32x2(k2, u01, make_float2(s[r].x, s[r].y));
                const float2 s23 = fma_f32x2(k2, u23, make_float2(s[r].z, s[r].w));
                s[r] = make_float4(s01.x, s01.y, s23.x, s23.y);
            }
            if (t + 1 == ncommit && S) {  // uniform: the stores issue only on the commit token
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    __stcs(reinterpret_cast<float4*>(S + (16 * warp + r) * kDim) + lane, s[r]);
            }
            __syncthreads();  // shared vectors are rewritten by the next token
        }
    }
}

}  // namespace

cudaError_t launch_decode_window(int dtype, int num_seqs, int heads, const void* q,
                                 const void* k, const void* v, const void* g, const void* beta,
                                 const int32_t* cu_seqlens, const float* state_in,
                                 float* state_out, void* out, const int32_t* commit,
                                 int64_t total_tokens, int max_len, int* status,
                                 cudaStream_t stream, const ProParams* pro) {
    const int64_t units = (int64_t)num_seqs * heads;
    if (units <= 0) return cudaSuccess;
    if (pro && dtype != KDA_BF16) return cudaErrorInvalidValue;
    using T = __nv_bfloat16;
    const DecPro dp = pro ? DecPro{pro->A_log, pro->dt_bias, pro->lower_bound, pro->q_scale, heads}
                          : DecPro{nullptr, nullptr, 0.f, 1.f, heads};
    auto kernel = pro ? kda_decode_window_kernel<T, true> : kda_decode_window_kernel<T, false>;
    // persistent grid: one CTA per resident slot, each taking units in strides of the grid
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess)
        err = dtype == KDA_BF16
                  ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDecodeThreads, 0)
                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &per_sm, kda_decode_window_kernel<float, false>, kDecodeThreads, 0);
    if (err != cudaSuccess) return err;
    const int64_t slots = (int64_t)(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(units < slots ? units : slots);
    if (dtype == KDA_BF16) {
        kernel<<<grid, kDecodeThreads, 0, stream>>>(
            (const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta, cu_seqlens,
            state_in, state_out, (T*)out, commit, units, heads, total_tokens, max_len, status, dp);
    } else {
        kda_decode_window_kernel<float, false><<<grid, kDecodeThreads, 0, stream>>>(
            (const float*)q, (const float*)k, (const float*)v, (const float*)g,
            (const float*)beta, cu_seqlens, state_in, state_out, (float*)out, commit, units,
            heads, total_tokens, max_len, status, dp);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode(int dtype, int64_t units, int heads, const void* q, const void* k,
                          const void* v, const void* g, const void* beta, float* state,
                          void* out, int* status, cudaStream_t stream, const ProParams* pro) {
    (void)status;
    if (units <= 0) return cudaSuccess;
    if (pro && dtype != KDA_BF16) return cudaErrorInvalidValue;
    const DecPro dp = pro ? DecPro{pro->A_log, pro->dt_bias, pro->lower_bound, pro->q_scale, heads}
                          : DecPro{nullptr, nullptr, 0.f, 1.f, heads};
    const int64_t max_grid = 1LL << 30;
    const unsigned grid = (unsigned)(units < max_grid ? units : max_grid);
    if (dtype == KDA_BF16) {
        using T = __nv_bfloat16;
        auto kernel = pro ? kda_decode_kernel<T, true> : kda_decode_kernel<T, false>;
        kernel<<<grid, kDecodeThreads, 0, stream>>>(
            (const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta, state, (T*)out,
            units, dp);
    } else {
        kda_decode_kernel<float, false><<<grid, kDecodeThreads, 0, stream>>>(
            (const float*)q, (const float*)k, (const float*)v, (const float*)g,
            (const float*)beta, state, (float*)out, units, dp);
    }
    return cudaGetLastError();
}

}  // namespace kda
