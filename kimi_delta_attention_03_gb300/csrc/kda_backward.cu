// kda_backward.cu — gradients of the KDA recurrence (the backward pass), on CUDA cores.
//
// Forward, per (sequence, head) unit and token t ("How Kimi K3 Engineered Its Way to the Frontier",
// section "How KDA updates its state"):
//     S' = diag(a_t) S,  a_t = exp(g_t);   r = v_t - S'^T k_t;   u = beta_t r;
//     S  <- S' + k_t u^T;                  o_t = S^T q_t
// Reverse mode, given dS (the gradient of the state after token t, carried backwards) and do_t:
//     dS += q_t do_t^T;     dq_t = S_t do_t = S' do_t + k_t (u . do_t)
//     du = dS^T k_t;        dv_t = beta_t du;      dbeta_t = du . r
//     dk_t = dS u - beta_t S' du
//     dS' = dS - beta_t k_t du^T;   dg_t = rowsum(dS' * S');   dS <- diag(a_t) dS'
// and the gradient of the initial state is dS after the first token.
//
// One CTA of 256 threads per unit; thread (warp w, lane l) holds rows {w + 8 r : r < 16} and
// columns 4l .. 4l+3 of S', and of dS, in registers (the decode step's layout).  A forward sweep
// stores the state before every 16-token block into the caller's workspace; the reverse sweep
// recomputes each block's states from its stored start (keeping the 16 of them in the workspace)
// and walks the block backwards.  Column sums go through shared memory, row sums through warp
// shuffles.  fp32 throughout.  This is a correctness-first kernel: it reads and writes 128 KB of
// workspace per token and unit, against the forward's chunked tensor-core path.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdBlock = 16;  // tokens per stored state

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Sixteen row sums across the warp at once (a reduce-scatter): halving exchanges over lane bits
// 0..3 leave each lane one partial of one row, and a last exchange over bit 4 completes it.  Lane
// l (and l + 16) ends with the sum for row index bitreverse4(l & 15).  16 shuffles instead of 80.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int half = 8 >> s;                 // values kept after this step
        const bool upper = (lane >> s) & 1;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << s);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}
__device__ __forceinline__ int bitrev4(int x) {
    return ((x & 1) << 3) | ((x & 2) << 1) | ((x & 4) >> 1) | ((x & 8) >> 3);
}

template <typename TIn>
struct BwdArgs {
    const TIn *q, *k, *v, *g, *beta;
    const int32_t* cu_seqlens;
    const float* init_state;  // [N][H][128][128] or null
    const float* d_out;       // [T][H][128]
    const float* d_state;     // [N][H][128][128] or null
    float *dq, *dk, *dv, *dg, *dbeta, *d_init;
    float* work;              // per unit: (nb_max + kBwdBlock) states of 128 x 128, then
                              // kBwdBlock pairs of 128-vectors (u, r)
    int64_t work_per_unit;    // floats
    int64_t total_tokens;     // host T_tot
    int* status;              // sticky status word
    int H;
};

template <typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 1) kda_bwd_kernel(const BwdArgs<TIn> p) {
    __shared__ float s_k[kDim], s_q[kDim], s_a[kDim], s_v[kDim], s_do[kDim];
    __shared__ float s_u[kDim], s_r[kDim], s_du[kDim];
    __shared__ __align__(16) float s_part[8][kDim];
    __shared__ float s_ud;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t unit = blockIdx.x;
    const int n = (int)(unit / p.H), h = (int)(unit - (int64_t)n * p.H);
    const int64_t t0 = p.cu_seqlens[n];
    const int L = (int)(p.cu_seqlens[n + 1] - t0);
    const int nb = (L + kBwdBlock - 1) / kBwdBlock;
    // The device cu_seqlens must agree with the host lengths the workspace was sized from: the
    // tokens stay inside T_tot and the unit's blocks inside its workspace region.
    if (t0 < 0 || L < 0 || t0 + L > p.total_tokens ||
        nb > (p.work_per_unit - kBwdBlock * 2 * kDim) / (kDim * kDim) - kBwdBlock) {
        if (tid == 0) report_status(p.status, KDA_ERR_INVALID_ARG);
        return;
    }
    float* ck = p.work + unit * p.work_per_unit;      // [nb][128 * 128]: state before block b
    float* blk = ck + (int64_t)nb * kDim * kDim;     // [kBwdBlock][128 * 128]: S' within a block
    float* blk_ur = p.work + unit * p.work_per_unit + p.work_per_unit - kBwdBlock * 2 * kDim;
    const int64_t sbase = unit * (int64_t)(kDim * kDim);

    auto ld_state = [&](const float* src, float4 (&x)[16]) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
            x[r] = src ? reinterpret_cast<const float4*>(src + (warp + 8 * r) * kDim)[lane]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto st_state = [&](float* dst, const float4 (&x)[16]) {
#pragma unroll
        for (int r = 0; r < 16; ++r) reinterpret_cast<float4*>(dst + (warp + 8 * r) * kDim)[lane] = x[r];
    };
    // One token's inputs, held raw in registers from their load to their staging, so that the next
    // token's loads are in flight while this one computes: k, g and v for a forward step; k, g,
    // q, d_out and the stored (u, r) for a reverse step (ur non-null).  Threads >= 128 load beta only.
    struct Tok {
        TIn k, g, v, q, b;
        float d, u, r;
    };
    auto fetch = [&](int t, const float* ur) -> Tok {
        Tok x;
        const int64_t row = (t0 + t) * p.H + h;
        x.b = p.beta[row];
        if (tid < kDim) {
            const int64_t e = row * kDim + tid;
            x.k = p.k[e];
            x.g = p.g[e];
            if (ur) {
                x.q = p.q[e];
                x.d = p.d_out[e];
                x.u = ur[tid];
                x.r = ur[kDim + tid];
            } else {
                x.v = p.v[e];
            }
        }
        return x;
    };
    // a fetched token into shared memory (a = exp(g)); returns its beta
    auto stage = [&](const Tok& x, bool reverse) -> float {
        if (tid < kDim) {
            s_k[tid] = io<TIn>::to_f(x.k);
            s_a[tid] = expf(io<TIn>::to_f(x.g));
            if (reverse) {
                s_q[tid] = io<TIn>::to_f(x.q);
                s_do[tid] = x.d;
                s_u[tid] = x.u;
                s_r[tid] = x.r;
            } else {
                s_v[tid] = io<TIn>::to_f(x.v);
            }
        }
        return io<TIn>::to_f(x.b);
    };
    // S' = diag(a) S in place, and the per-warp partial column sums of k_i S'_ij into s_part
    auto decay_and_x = [&](float4 (&S)[16]) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = warp + 8 * r;
            const float a = s_a[i], kk = s_k[i];
            S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
            x.x = fmaf(kk, S[r].x, x.x); x.y = fmaf(kk, S[r].y, x.y);
            x.z = fmaf(kk, S[r].z, x.z); x.w = fmaf(kk, S[r].w, x.w);
        }
        reinterpret_cast<float4*>(s_part[warp])[lane] = x;
    };
    // r = v - S'^T k and u = beta r into s_r, s_u (threads < 128), and into keep_ur when given
    auto make_u = [&](float b, float* keep_ur) {
        if (tid < kDim) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) x += s_part[w][tid];
            const float r = s_v[tid] - x;
            s_r[tid] = r;
            s_u[tid] = b * r;
            if (keep_ur) {
                keep_ur[tid] = b * r;
                keep_ur[kDim + tid] = r;
            }
        }
    };
    // one forward token: S <- diag(a) S + k u^T; keeps S' = diag(a) S and (u, r) when asked
    // nx holds token t's inputs on entry and token t_next's (when t_next >= 0) on return
    auto fwd_step = [&](float4 (&S)[16], float* keep_s, float* keep_ur, Tok& nx, int t_next) {
        const float b = stage(nx, false);
        if (t_next >= 0) nx = fetch(t_next, nullptr);
        __syncthreads();
        decay_and_x(S);
        if (keep_s) st_state(keep_s, S);
        __syncthreads();
        make_u(b, keep_ur);
        __syncthreads();
        const float4 u4 = reinterpret_cast<const float4*>(s_u)[lane];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float kk = s_k[warp + 8 * r];
            S[r].x = fmaf(kk, u4.x, S[r].x); S[r].y = fmaf(kk, u4.y, S[r].y);
            S[r].z = fmaf(kk, u4.z, S[r].z); S[r].w = fmaf(kk, u4.w, S[r].w);
        }
        __syncthreads();  // the shared vectors are rewritten by the next token
    };

    float4 S[16], dS[16];
    // ---- forward sweep: the state before every block
    ld_state(p.init_state ? p.init_state + sbase : nullptr, S);
    Tok nx;
    if (L > 0) nx = fetch(0, nullptr);
#pragma unroll 1
    for (int b = 0; b < nb; ++b) {
        st_state(ck + (int64_t)b * kDim * kDim, S);
        const int te = min(L, (b + 1) * kBwdBlock);
#pragma unroll 1
        for (int t = b * kBwdBlock; t < te; ++t) fwd_step(S, nullptr, nullptr, nx, t + 1 < L ? t + 1 : -1);
    }
    // ---- reverse sweep
    ld_state(p.d_state ? p.d_state + sbase : nullptr, dS);
#pragma unroll 1
    for (int b = nb - 1; b >= 0; --b) {
        const int tb = b * kBwdBlock, te = min(L, tb + kBwdBlock);
        __syncthreads();  // this block's stored states are rewritten below
        ld_state(ck + (int64_t)b * kDim * kDim, S);
        nx = fetch(tb, nullptr);
#pragma unroll 1
        for (int t = tb; t < te; ++t)
            fwd_step(S, blk + (int64_t)(t - tb) * kDim * kDim, blk_ur + (t - tb) * 2 * kDim, nx,
                     t + 1 < te ? t + 1 : -1);
        // the (u, r) a reverse step fetches were written by this thread in the replay above
        nx = fetch(te - 1, blk_ur + (te - 1 - tb) * 2 * kDim);
#pragma unroll 1
        for (int t = te - 1; t >= tb; --t) {
            const int64_t row = (t0 + t) * p.H + h;
            ld_state(blk + (int64_t)(t - tb) * kDim * kDim, S);  // S' = diag(a_t) S_{t-1}
            const float b_t = stage(nx, true);
            if (t > tb) nx = fetch(t - 1, blk_ur + (t - 1 - tb) * 2 * kDim);
            __syncthreads();
            // dS += q do^T; partial column sums of k_i dS_ij; u . do
            {
                const float4 do4 = reinterpret_cast<const float4*>(s_do)[lane];
                float4 dup = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const int i = warp + 8 * r;
                    const float qq = s_q[i], kk = s_k[i];
                    dS[r].x = fmaf(qq, do4.x, dS[r].x); dS[r].y = fmaf(qq, do4.y, dS[r].y);
                    dS[r].z = fmaf(qq, do4.z, dS[r].z); dS[r].w = fmaf(qq, do4.w, dS[r].w);
                    dup.x = fmaf(kk, dS[r].x, dup.x); dup.y = fmaf(kk, dS[r].y, dup.y);
                    dup.z = fmaf(kk, dS[r].z, dup.z); dup.w = fmaf(kk, dS[r].w, dup.w);
                }
                reinterpret_cast<float4*>(s_part[warp])[lane] = dup;
                if (warp == 0) {
                    const float4 u4 = reinterpret_cast<const float4*>(s_u)[lane];
                    const float ud = warp_sum(u4.x * do4.x + u4.y * do4.y + u4.z * do4.z + u4.w * do4.w);
                    if (lane == 0) s_ud = ud;
                }
            }
            __syncthreads();
            if (tid < kDim) {  // du = dS^T k; dv = beta du
                float du = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) du += s_part[w][tid];
                s_du[tid] = du;
                p.dv[row * kDim + tid] = b_t * du;
            }
            __syncthreads();
            {
                const float4 du4 = reinterpret_cast<const float4*>(s_du)[lane];
                const float4 u4 = reinterpret_cast<const float4*>(s_u)[lane];
                const float4 do4 = reinterpret_cast<const float4*>(s_do)[lane];
                const float ud = s_ud;
                if (warp == 0) {  // dbeta = du . r
                    const float4 r4 = reinterpret_cast<const float4*>(s_r)[lane];
                    const float db = warp_sum(du4.x * r4.x + du4.y * r4.y + du4.z * r4.z + du4.w * r4.w);
                    if (lane == 0) p.dbeta[row] = db;
                }
                // row sums in three passes of 16 (one per gradient), each a warp reduce-scatter
                const int rr = bitrev4(lane & 15);  // the row (of this warp's 16) this lane ends with
                float part[16];
#pragma unroll
                for (int r = 0; r < 16; ++r)  // dq_i = (S' do)_i + k_i (u . do)
                    part[r] = S[r].x * do4.x + S[r].y * do4.y + S[r].z * do4.z + S[r].w * do4.w;
                {
                    const float sum = warp_sum16(part, lane);
                    const int i = warp + 8 * rr;
                    if (lane < 16) p.dq[row * kDim + i] = fmaf(s_k[i], ud, sum);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r)  // dk_i = (dS u)_i - beta (S' du)_i
                    part[r] = dS[r].x * u4.x + dS[r].y * u4.y + dS[r].z * u4.z + dS[r].w * u4.w -
                              b_t * (S[r].x * du4.x + S[r].y * du4.y + S[r].z * du4.z + S[r].w * du4.w);
                {
                    const float sum = warp_sum16(part, lane);
                    if (lane < 16) p.dk[row * kDim + warp + 8 * rr] = sum;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {  // dS' = dS - beta k du^T; dg_i = rowsum(dS' * S')
                    const float bk = b_t * s_k[warp + 8 * r];
                    dS[r].x = fmaf(-bk, du4.x, dS[r].x); dS[r].y = fmaf(-bk, du4.y, dS[r].y);
                    dS[r].z = fmaf(-bk, du4.z, dS[r].z); dS[r].w = fmaf(-bk, du4.w, dS[r].w);
                    part[r] = dS[r].x * S[r].x + dS[r].y * S[r].y + dS[r].z * S[r].z + dS[r].w * S[r].w;
                    const float a = s_a[warp + 8 * r];  // dS <- diag(a) dS'
                    dS[r].x *= a; dS[r].y *= a; dS[r].z *= a; dS[r].w *= a;
                }
                {
                    const float sum = warp_sum16(part, lane);
                    if (lane < 16) p.dg[row * kDim + warp + 8 * rr] = sum;
                }
            }
            __syncthreads();  // the shared vectors are rewritten by the previous token
        }
    }
    st_state(p.d_init + sbase, dS);
}

}  // namespace

cudaError_t launch_backward(int dtype, int num_seqs, int heads, const void* q, const void* k,
                            const void* v, const void* g, const void* beta,
                            const int32_t* cu_seqlens, const float* init_state,
                            const float* d_out, const float* d_state, float* dq, float* dk,
                            float* dv, float* dg, float* dbeta, float* d_init, float* work,
                            int64_t work_per_unit, int64_t total_tokens, int* status,
                            cudaStream_t stream) {
    const int64_t units = (int64_t)num_seqs * heads;
    if (units <= 0) return cudaSuccess;
    if (dtype == KDA_BF16) {
        using T = __nv_bfloat16;
        const BwdArgs<T> a{(const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta,
                           cu_seqlens, init_state, d_out, d_state, dq, dk, dv, dg, dbeta, d_init,
                           work, work_per_unit, total_tokens, status, heads};
        kda_bwd_kernel<T><<<(unsigned)units, kBwdThreads, 0, stream>>>(a);
    } else {
        const BwdArgs<float> a{(const float*)q, (const float*)k, (const float*)v, (const float*)g,
                               (const float*)beta, cu_seqlens, init_state, d_out, d_state, dq,
                               dk, dv, dg, dbeta, d_init, work, work_per_unit, total_tokens, status,
                               heads};
        kda_bwd_kernel<float><<<(unsigned)units, kBwdThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
