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
// The value channels (columns of S) evolve independently: x = S'^T k, u, du = dS^T k and the
// updates of S and dS act column by column, so each unit runs as kBwdColBlocks CTAs of 128
// threads, one per block of kDim / kBwdColBlocks columns.  Only the outputs dq, dk, dg and dbeta
// sum over the columns; each CTA writes its block's partial sums into the workspace, and a second
// launch adds the partials in a fixed order, so the gradients do not depend on scheduling.
//
// Thread t of a CTA holds one float4 of columns (t % kLanesPerRow) and rows
// {t / kLanesPerRow + kRowGroups r} of S', and of dS, in registers (with 32-column blocks a warp
// covers four consecutive rows of 32 columns per access).  A forward sweep stores the state
// before every 16-token block into the caller's workspace; the reverse sweep recomputes each
// block's states from its stored start (keeping the 16 of them in the workspace) and walks the
// block backwards.  Column sums and row sums go through shared memory.  fp32 throughout, on CUDA
// cores.
#include <algorithm>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdBlock = 16;   // tokens per stored state
constexpr int kCols = kDim / kBwdColBlocks;          // columns per CTA
constexpr int kLanesPerRow = kCols / 4;                 // lanes that share a row (a float4 each)
constexpr int kRowGroups = kBwdThreads / kLanesPerRow;  // rows held at once by the CTA
constexpr int kRowsPer = kDim / kRowGroups;             // rows of S per thread
constexpr int kColBlocks = kBwdColBlocks;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <typename TIn>
struct BwdArgs {
    const TIn *q, *k, *v, *g, *beta;
    const int32_t* cu_seqlens;
    const float* init_state;  // [N][H][128][128] or null
    const float* d_out;       // [T][H][128]
    const float* d_state;     // [N][H][128][128] or null
    float *dv, *d_init;       // written directly
    float* part;              // [3][kColBlocks][T][H][128] partial dq, dk, dg, then
                              // [kColBlocks][T][H] partial dbeta
    float* work;              // per (unit, column block): (nb_max + kBwdBlock) states of
                              // 128 x 32, then kBwdBlock pairs of 32-vectors (u, r)
    int64_t work_per_cta;     // floats
    int64_t total_tokens;     // host T_tot
    int* status;              // sticky status word
    int H;
};

template <typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 4) kda_bwd_kernel(const BwdArgs<TIn> p) {
    __shared__ float s_k[kDim], s_q[kDim], s_a[kDim];
    __shared__ float s_v[kCols], s_do[kCols], s_u[kCols], s_r[kCols], s_du[kCols];
    __shared__ __align__(16) float s_part[kRowGroups][kCols];       // per row group, column partials
    __shared__ __align__(16) float s_rp[3][kDim][kLanesPerRow];     // per row, 4-column partials
    __shared__ float s_ud;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cq = tid % kLanesPerRow;        // float4 column group within the block
    const int rg = tid / kLanesPerRow;        // row group: rows rg + kRowGroups r
    const int64_t unit = blockIdx.x / kColBlocks;
    const int cb = (int)(blockIdx.x - unit * kColBlocks);
    const int j0 = cb * kCols;                // first column of this CTA
    const int n = (int)(unit / p.H), h = (int)(unit - (int64_t)n * p.H);
    const int64_t t0 = p.cu_seqlens[n];
    const int L = (int)(p.cu_seqlens[n + 1] - t0);
    const int nb = (L + kBwdBlock - 1) / kBwdBlock;
    // The device cu_seqlens must agree with the host lengths the workspace was sized from: the
    // tokens stay inside T_tot and the unit's blocks inside its workspace region.  Every CTA of
    // the unit takes the same decision.
    if (t0 < 0 || L < 0 || t0 + L > p.total_tokens ||
        nb > (p.work_per_cta - kBwdBlock * 2 * kCols) / (kDim * kCols) - kBwdBlock) {
        if (tid == 0) report_status(p.status, KDA_ERR_INVALID_ARG);
        return;
    }
    float* ck = p.work + (unit * kColBlocks + cb) * p.work_per_cta;  // [nb][128 * 32]
    float* blk = ck + (int64_t)nb * kDim * kCols;                      // [16][128 * 32]
    float* blk_ur = ck + p.work_per_cta - kBwdBlock * 2 * kCols;       // [16][2][32]
    const int64_t sbase = unit * (int64_t)(kDim * kDim);
    const int64_t TH = p.total_tokens * p.H;
    float* pdq = p.part + (int64_t)cb * TH * kDim;
    float* pdk = p.part + (int64_t)(kColBlocks + cb) * TH * kDim;
    float* pdg = p.part + (int64_t)(2 * kColBlocks + cb) * TH * kDim;
    float* pdb = p.part + (int64_t)3 * kColBlocks * TH * kDim + (int64_t)cb * TH;

    // a full [128][128] state (columns j0 .. j0 + 31) or a compact [128][32] one
    auto ld_full = [&](const float* src, float4 (&x)[kRowsPer]) {
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r)
            x[r] = src ? reinterpret_cast<const float4*>(src + (rg + kRowGroups * r) * kDim + j0)[cq]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto ld_blk = [&](const float* src, float4 (&x)[kRowsPer]) {
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r)
            x[r] = reinterpret_cast<const float4*>(src + (rg + kRowGroups * r) * kCols)[cq];
    };
    auto st_blk = [&](float* dst, const float4 (&x)[kRowsPer]) {
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r)
            reinterpret_cast<float4*>(dst + (rg + kRowGroups * r) * kCols)[cq] = x[r];
    };
    // One token's inputs, held raw in registers from their load to their staging, so that the
    // next token's loads are in flight while this one computes: k, g (row tid) and v (column
    // j0 + tid, tid < 32) for a forward step; also q (row tid), d_out and the stored (u, r)
    // (tid < 32) for a reverse step (ur non-null).
    struct Tok {
        TIn k, g, v, q, b;
        float d, u, r;
    };
    auto fetch = [&](int t, const float* ur) -> Tok {
        Tok x;
        const int64_t row = (t0 + t) * p.H + h;
        x.b = p.beta[row];
        const int64_t e = row * kDim + tid;
        x.k = p.k[e];
        x.g = p.g[e];
        if (ur) {
            x.q = p.q[e];
            if (tid < kCols) {
                x.d = p.d_out[row * kDim + j0 + tid];
                x.u = ur[tid];
                x.r = ur[kCols + tid];
            }
        } else if (tid < kCols) {
            x.v = p.v[row * kDim + j0 + tid];
        }
        return x;
    };
    // a fetched token into shared memory (a = exp(g)); returns its beta
    auto stage = [&](const Tok& x, bool reverse) -> float {
        s_k[tid] = io<TIn>::to_f(x.k);
        s_a[tid] = expf(io<TIn>::to_f(x.g));
        if (reverse) {
            s_q[tid] = io<TIn>::to_f(x.q);
            if (tid < kCols) {
                s_do[tid] = x.d;
                s_u[tid] = x.u;
                s_r[tid] = x.r;
            }
        } else if (tid < kCols) {
            s_v[tid] = io<TIn>::to_f(x.v);
        }
        return io<TIn>::to_f(x.b);
    };
    // one forward token: S' = diag(a) S; x = S'^T k; r = v - x; u = beta r; S <- S' + k u^T.
    // Keeps S' and (u, r) when asked; nx holds token t's inputs on entry and token t_next's
    // (when t_next >= 0) on return.
    auto fwd_step = [&](float4 (&S)[kRowsPer], float* keep_s, float* keep_ur, Tok& nx,
                        int t_next) {
        const float b = stage(nx, false);
        if (t_next >= 0) nx = fetch(t_next, nullptr);
        __syncthreads();
        {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < kRowsPer; ++r) {
                const int i = rg + kRowGroups * r;
                const float a = s_a[i], kk = s_k[i];
                S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
                x.x = fmaf(kk, S[r].x, x.x); x.y = fmaf(kk, S[r].y, x.y);
                x.z = fmaf(kk, S[r].z, x.z); x.w = fmaf(kk, S[r].w, x.w);
            }
            reinterpret_cast<float4*>(s_part[rg])[cq] = x;
            if (keep_s) st_blk(keep_s, S);
        }
        __syncthreads();
        if (tid < kCols) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < kRowGroups; ++w) x += s_part[w][tid];
            const float r = s_v[tid] - x;
            s_r[tid] = r;
            s_u[tid] = b * r;
            if (keep_ur) {
                keep_ur[tid] = b * r;
                keep_ur[kCols + tid] = r;
            }
        }
        __syncthreads();
        const float4 u4 = reinterpret_cast<const float4*>(s_u)[cq];
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r) {
            const float kk = s_k[rg + kRowGroups * r];
            S[r].x = fmaf(kk, u4.x, S[r].x); S[r].y = fmaf(kk, u4.y, S[r].y);
            S[r].z = fmaf(kk, u4.z, S[r].z); S[r].w = fmaf(kk, u4.w, S[r].w);
        }
        __syncthreads();  // the shared vectors are rewritten by the next token
    };

    float4 S[kRowsPer], dS[kRowsPer];
    // ---- forward sweep: the state before every block
    ld_full(p.init_state ? p.init_state + sbase : nullptr, S);
    Tok nx;
    if (L > 0) nx = fetch(0, nullptr);
#pragma unroll 1
    for (int b = 0; b < nb; ++b) {
        st_blk(ck + (int64_t)b * kDim * kCols, S);
        const int te = min(L, (b + 1) * kBwdBlock);
#pragma unroll 1
        for (int t = b * kBwdBlock; t < te; ++t)
            fwd_step(S, nullptr, nullptr, nx, t + 1 < L ? t + 1 : -1);
    }
    // ---- reverse sweep
    ld_full(p.d_state ? p.d_state + sbase : nullptr, dS);
#pragma unroll 1
    for (int b = nb - 1; b >= 0; --b) {
        const int tb = b * kBwdBlock, te = min(L, tb + kBwdBlock);
        __syncthreads();  // this block's stored states are rewritten below
        ld_blk(ck + (int64_t)b * kDim * kCols, S);
        nx = fetch(tb, nullptr);
#pragma unroll 1
        for (int t = tb; t < te; ++t)
            fwd_step(S, blk + (int64_t)(t - tb) * kDim * kCols, blk_ur + (t - tb) * 2 * kCols, nx,
                     t + 1 < te ? t + 1 : -1);
        // the (u, r) a reverse step fetches were written by this thread in the replay above
        nx = fetch(te - 1, blk_ur + (te - 1 - tb) * 2 * kCols);
#pragma unroll 1
        for (int t = te - 1; t >= tb; --t) {
            const int64_t row = (t0 + t) * p.H + h;
            ld_blk(blk + (int64_t)(t - tb) * kDim * kCols, S);  // S' = diag(a_t) S_{t-1}
            const float k_own = io<TIn>::to_f(nx.k);            // k of row tid
            const float b_t = stage(nx, true);
            if (t > tb) nx = fetch(t - 1, blk_ur + (t - 1 - tb) * 2 * kCols);
            __syncthreads();
            // dS += q do^T; column partials of k_i dS_ij; u . do over this block's columns
            {
                const float4 do4 = reinterpret_cast<const float4*>(s_do)[cq];
                float4 dup = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int r = 0; r < kRowsPer; ++r) {
                    const int i = rg + kRowGroups * r;
                    const float qq = s_q[i], kk = s_k[i];
                    dS[r].x = fmaf(qq, do4.x, dS[r].x); dS[r].y = fmaf(qq, do4.y, dS[r].y);
                    dS[r].z = fmaf(qq, do4.z, dS[r].z); dS[r].w = fmaf(qq, do4.w, dS[r].w);
                    dup.x = fmaf(kk, dS[r].x, dup.x); dup.y = fmaf(kk, dS[r].y, dup.y);
                    dup.z = fmaf(kk, dS[r].z, dup.z); dup.w = fmaf(kk, dS[r].w, dup.w);
                }
                reinterpret_cast<float4*>(s_part[rg])[cq] = dup;
                if (warp == 0) {  // every lane takes part; lanes past the block's columns add 0
                    const float ud = warp_sum(lane < kCols ? s_u[lane] * s_do[lane] : 0.f);
                    if (lane == 0) s_ud = ud;
                }
            }
            __syncthreads();
            if (warp == 0) {  // du = dS^T k; dv = beta du; dbeta partial = du . r
                float dr = 0.f;
                if (lane < kCols) {
                    float du = 0.f;
#pragma unroll
                    for (int w = 0; w < kRowGroups; ++w) du += s_part[w][lane];
                    s_du[lane] = du;
                    p.dv[row * kDim + j0 + lane] = b_t * du;
                    dr = du * s_r[lane];
                }
                const float db = warp_sum(dr);  // every lane of warp 0 takes part
                if (lane == 0) pdb[row] = db;
            }
            __syncthreads();
            const float ud = s_ud;
            {
                const float4 du4 = reinterpret_cast<const float4*>(s_du)[cq];
                const float4 u4 = reinterpret_cast<const float4*>(s_u)[cq];
                const float4 do4 = reinterpret_cast<const float4*>(s_do)[cq];
#pragma unroll
                for (int r = 0; r < kRowsPer; ++r) {
                    const int i = rg + kRowGroups * r;
                    // dq_i = (S' do)_i + k_i (u . do); dk_i = (dS u)_i - beta (S' du)_i
                    s_rp[0][i][cq] = S[r].x * do4.x + S[r].y * do4.y + S[r].z * do4.z + S[r].w * do4.w;
                    s_rp[1][i][cq] = dS[r].x * u4.x + dS[r].y * u4.y + dS[r].z * u4.z + dS[r].w * u4.w -
                                     b_t * (S[r].x * du4.x + S[r].y * du4.y + S[r].z * du4.z + S[r].w * du4.w);
                    // dS' = dS - beta k du^T; dg_i = rowsum(dS' * S'); dS <- diag(a) dS'
                    const float bk = b_t * s_k[i];
                    dS[r].x = fmaf(-bk, du4.x, dS[r].x); dS[r].y = fmaf(-bk, du4.y, dS[r].y);
                    dS[r].z = fmaf(-bk, du4.z, dS[r].z); dS[r].w = fmaf(-bk, du4.w, dS[r].w);
                    s_rp[2][i][cq] = dS[r].x * S[r].x + dS[r].y * S[r].y + dS[r].z * S[r].z + dS[r].w * S[r].w;
                    const float a = s_a[i];
                    dS[r].x *= a; dS[r].y *= a; dS[r].z *= a; dS[r].w *= a;
                }
            }
            __syncthreads();
            {  // this block's partial row sums for row tid (read before the next token's barrier)
                float sq = 0.f, sk = 0.f, sg = 0.f;
#pragma unroll
                for (int e = 0; e < kLanesPerRow; ++e) {
                    sq += s_rp[0][tid][e];
                    sk += s_rp[1][tid][e];
                    sg += s_rp[2][tid][e];
                }
                pdq[row * kDim + tid] = fmaf(k_own, ud, sq);
                pdk[row * kDim + tid] = sk;
                pdg[row * kDim + tid] = sg;
            }
        }
    }
    // d_init: this block's columns of dS after the first token
    {
        float* dst = p.d_init + sbase;
#pragma unroll
        for (int r = 0; r < kRowsPer; ++r)
            reinterpret_cast<float4*>(dst + (rg + kRowGroups * r) * kDim + j0)[cq] = dS[r];
    }
}

// dq, dk, dg and dbeta: the sums of the column blocks' partials, in block order.
__global__ void __launch_bounds__(256) kda_bwd_sum_kernel(const float* __restrict__ part,
                                                         int64_t TH, float* __restrict__ dq,
                                                         float* __restrict__ dk,
                                                         float* __restrict__ dg,
                                                         float* __restrict__ dbeta) {
    const int64_t n4 = TH * kDim / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < 3 * n4 + TH; e += stride) {
        if (e < 3 * n4) {
            const int which = (int)(e / n4);
            const int64_t i = e - which * n4;
            const float4* src = reinterpret_cast<const float4*>(part) + (int64_t)which * kColBlocks * n4 + i;
            float4 acc = src[0];
#pragma unroll
            for (int c = 1; c < kColBlocks; ++c) {
                const float4 x = src[c * n4];
                acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
            }
            float* o = which == 0 ? dq : which == 1 ? dk : dg;
            reinterpret_cast<float4*>(o)[i] = acc;
        } else {
            const int64_t i = e - 3 * n4;
            const float* src = part + 3 * kColBlocks * TH * kDim + i;
            float acc = src[0];
#pragma unroll
            for (int c = 1; c < kColBlocks; ++c) acc += src[c * TH];
            dbeta[i] = acc;
        }
    }
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
    // the units' state regions, then the partial sums
    float* part = work + units * work_per_unit;
    const int64_t per_cta = work_per_unit / kColBlocks;
    const unsigned grid = (unsigned)(units * kColBlocks);
    if (dtype == KDA_BF16) {
        using T = __nv_bfloat16;
        const BwdArgs<T> a{(const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta,
                           cu_seqlens, init_state, d_out, d_state, dv, d_init, part, work,
                           per_cta, total_tokens, status, heads};
        kda_bwd_kernel<T><<<grid, kBwdThreads, 0, stream>>>(a);
    } else {
        const BwdArgs<float> a{(const float*)q, (const float*)k, (const float*)v, (const float*)g,
                               (const float*)beta, cu_seqlens, init_state, d_out, d_state, dv,
                               d_init, part, work, per_cta, total_tokens, status, heads};
        kda_bwd_kernel<float><<<grid, kBwdThreads, 0, stream>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t TH = total_tokens * heads;
    if (TH > 0) {
        const int64_t items = 3 * TH * kDim / 4 + TH;
        const unsigned blocks = (unsigned)std::min<int64_t>((items + 255) / 256, 152 * 16);
        kda_bwd_sum_kernel<<<blocks, 256, 0, stream>>>(part, TH, dq, dk, dg, dbeta);
    }
    return cudaGetLastError();
}

}  // namespace kda
