// kda_backward.cu — gradients of the KDA recurrence (the backward pass), chunked, on tensor cores.
//
// Forward, per (sequence, head) unit and token t ("How Kimi K3 Engineered Its Way to the Frontier",
// section "How KDA updates its state"):
//     S' = diag(exp g_t) S;   u_t = beta_t (v_t - S'^T k_t);   S <- S' + k_t u_t^T;   o_t = S^T q_t
// The backward steps the state once per 16-token chunk, as the pages' kernel does ("FlashKDA steps
// the state once per 16 tokens"): a chunk with start state S, end state S+ and chunk-local
//     G = cumsum g (per key channel), a = exp(G_C), r = G_C / 2
//     K_f = k e^G, Q_f = q e^G, K_bar = k e^(G_C - G), K_p = k e^(G - r), K_m = k e^(r - G),
//     Q_r = q e^(G - r)
//     At = strict_lower(K_p K_m^T), P = lower_incl(Q_r K_m^T), T = (I + diag(beta) At)^-1
//     R = V - K_f S,  U = T diag(beta) R,  O = Q_f S + P U,  S+ = diag(a) S + K_bar^T U
// has, for dE the gradient of S+ and dO that of O,
//     dU = P^T dO + K_bar dE,   dY = T^T dU,   dR = diag(beta) dY   (= dv)
//     dbeta = rowsum(dY * R) + rowsum(dA * At),   dA = -strict_lower(dY U^T),  dP = lower_incl(dO U^T)
//     dK_f = -dR S^T, dQ_f = dO S^T, dK_bar = U dE^T, dK_p = diag(beta) dA K_m,
//     dK_m = (diag(beta) dA)^T K_p + dP^T Q_r, dQ_r = dP K_m
//     dk = dK_f e^G + dK_p e^(G-r) + dK_m e^(r-G) + dK_bar e^(G_C-G);  dq = dQ_f e^G + dQ_r e^(G-r)
//     dG = k (dK_f e^G + dK_p e^(G-r) - dK_m e^(r-G) - dK_bar e^(G_C-G)) + q (dQ_f e^G + dQ_r e^(G-r))
//     dG[last] += sum_t dK_bar K_bar + a * rowsum(dE * S);   dg = suffix sum of dG over the chunk
//     dS = diag(a) dE + Q_f^T dO - K_f^T dR = diag(a) dE + Q_f^T dO - W^T dU,   W = T diag(beta) K_f
// The mid-chunk reference r keeps every factor within exp(+-80) when a 16-token chunk decays by at
// most 160 in every channel (a mean of -10 per token, twice the bounded gate's floor of -5).
// Exponentials use the fast hardware form (__expf): its relative error, about 1e-5 at |x| = 80,
// is far below the tf32 rounding (5e-4) that every factor then goes through.
//
// Four launches:
//   index   one CTA: chunk offsets of the sequences from the device cu_seqlens, checked against the
//           host's chunk total (a disagreement stops the later launches and reports it)
//   prep    one CTA per (chunk, head): At, P and T (16 x 16 each) into the workspace
//   forward one CTA per unit: the forward state chain, S^T kept in registers (warp w holds value
//           channels 16w..16w+15), writing each chunk's start state (fp32) into the workspace
//   reverse one CTA per unit: chunks in reverse, dE^T in shared memory, every gradient of the chunk
// All products are m16n8k8 tf32 mma.sync with fp32 accumulation: 16-token tiles are the shape of
// these instructions, and tf32 operands keep the gradients inside the parity gate where bf16
// operands do not.  Within an 8-wide k step, MMA slots t and t + 4 take columns 2t and 2t + 1, so
// that accumulator fragments feed the next product's A operand directly and operand pairs load as
// 64-bit words.  Shared tiles of 128 fp32 columns use an XOR swizzle that keeps both fragment
// access patterns (rows g, columns 2t..2t+1 and rows 2t, 2t+1, columns g) free of bank conflicts.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int kBC = 16;           // tokens per backward chunk
constexpr int kBwdChainThreads = 256;
constexpr int kPrepThreads = 128;
constexpr int kTile = kBC * kDim;      // floats in a [16][128] tile
constexpr int kState = kDim * kDim;    // floats in a state
constexpr int kSlot = kState + kTile;  // per chunk and head: S^T at the chunk's start, then R
constexpr int kSmallLd = 20;           // leading dimension of the 16 x 16 tiles in shared memory
constexpr int kSmall = kBC * kSmallLd;
constexpr float kMaxExponent = 80.f;   // |G - r| bound of the factors
constexpr long long kBwdWaitLimit = 4000000000LL;   // clock cycles (about 2 s)

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(tf32_bits(x)); }
__device__ __forceinline__ uint32_t bits(float x) { return __float_as_uint(x); }
__device__ __forceinline__ uint32_t neg(uint32_t x) { return x ^ 0x80000000u; }

__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Element (r, c) of a [rows][128] fp32 tile: columns XORed with 8 * ((r & 3) ^ ((r >> 2) & 1)).
__device__ __forceinline__ int swz(int r, int c) {
    return r * kDim + (c ^ ((((r & 3) ^ ((r >> 2) & 1))) << 3));
}

// A fragment (16 x 8, permuted k) of a row-major tile X[m][k]: rows m0+g, m0+g+8, columns
// k0+2t, k0+2t+1.
__device__ __forceinline__ void lda_mk(const float* s, int m0, int k0, int g, int t,
                                       uint32_t (&a)[4]) {
    const float2 lo = *reinterpret_cast<const float2*>(s + swz(m0 + g, k0 + 2 * t));
    const float2 hi = *reinterpret_cast<const float2*>(s + swz(m0 + g + 8, k0 + 2 * t));
    a[0] = bits(lo.x); a[1] = bits(hi.x); a[2] = bits(lo.y); a[3] = bits(hi.y);
}
// A fragment of A[m][k] = X[k][m] (the tile holds the transpose).
__device__ __forceinline__ void lda_km(const float* s, int m0, int k0, int g, int t,
                                       uint32_t (&a)[4]) {
    a[0] = bits(s[swz(k0 + 2 * t, m0 + g)]);
    a[1] = bits(s[swz(k0 + 2 * t, m0 + g + 8)]);
    a[2] = bits(s[swz(k0 + 2 * t + 1, m0 + g)]);
    a[3] = bits(s[swz(k0 + 2 * t + 1, m0 + g + 8)]);
}
// B fragment (8 x 8, permuted k) of B[k][n] = X[n][k].
__device__ __forceinline__ void ldb_nk(const float* s, int n0, int k0, int g, int t,
                                       uint32_t (&b)[2]) {
    const float2 v = *reinterpret_cast<const float2*>(s + swz(n0 + g, k0 + 2 * t));
    b[0] = bits(v.x); b[1] = bits(v.y);
}
// B fragment of B[k][n] = X[k][n].
__device__ __forceinline__ void ldb_kn(const float* s, int k0, int n0, int g, int t,
                                       uint32_t (&b)[2]) {
    b[0] = bits(s[swz(k0 + 2 * t, n0 + g)]);
    b[1] = bits(s[swz(k0 + 2 * t + 1, n0 + g)]);
}
// Accumulator rows m0+g, m0+g+8 and columns c0+2t, c0+2t+1 into a swizzled tile.
__device__ __forceinline__ void st_c(float* s, int m0, int c0, int g, int t, const float (&d)[4]) {
    *reinterpret_cast<float2*>(s + swz(m0 + g, c0 + 2 * t)) = make_float2(d[0], d[1]);
    *reinterpret_cast<float2*>(s + swz(m0 + g + 8, c0 + 2 * t)) = make_float2(d[2], d[3]);
}
// The same for the 16 x 16 tiles (leading dimension kSmallLd, no swizzle).
__device__ __forceinline__ void lda_small(const float* s, int k0, int g, int t, uint32_t (&a)[4]) {
    const float2 lo = *reinterpret_cast<const float2*>(s + g * kSmallLd + k0 + 2 * t);
    const float2 hi = *reinterpret_cast<const float2*>(s + (g + 8) * kSmallLd + k0 + 2 * t);
    a[0] = bits(lo.x); a[1] = bits(hi.x); a[2] = bits(lo.y); a[3] = bits(hi.y);
}
__device__ __forceinline__ void lda_small_tr(const float* s, int k0, int g, int t,
                                             uint32_t (&a)[4]) {
    a[0] = bits(s[(k0 + 2 * t) * kSmallLd + g]);
    a[1] = bits(s[(k0 + 2 * t) * kSmallLd + g + 8]);
    a[2] = bits(s[(k0 + 2 * t + 1) * kSmallLd + g]);
    a[3] = bits(s[(k0 + 2 * t + 1) * kSmallLd + g + 8]);
}

// One channel of a chunk: out[i] = x[(t0 + i) * H + h][ch] for i < nt, zero beyond.  The row
// index is clamped rather than branched on, so that all 16 loads are in flight together.
template <typename TIn>
__device__ __forceinline__ void load_col(const TIn* x, int64_t t0, int nt, int H, int h, int ch,
                                         float (&out)[kBC]) {
    TIn raw[kBC];
#pragma unroll
    for (int i = 0; i < kBC; ++i) raw[i] = x[((t0 + (i < nt ? i : nt - 1)) * H + h) * kDim + ch];
#pragma unroll
    for (int i = 0; i < kBC; ++i) out[i] = i < nt ? io<TIn>::to_f(raw[i]) : 0.f;
}

// Four consecutive channels of one row: their raw bits (8 bytes of bf16, 16 of fp32) and fp32.
template <typename TIn> struct Vec4;
template <> struct Vec4<__nv_bfloat16> {
    using T = uint2;
    static __device__ __forceinline__ float4 unpack(uint2 v) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};
template <> struct Vec4<float> {
    using T = uint4;
    static __device__ __forceinline__ float4 unpack(uint4 v) {
        return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                           __uint_as_float(v.w));
    }
};
// Rows t0 .. t0 + 15 (the last valid row repeated past nt) of channels 4 lane .. 4 lane + 3.
template <typename TIn>
__device__ __forceinline__ void load_rows4(const TIn* x, int64_t t0, int nt, int H, int h,
                                           int lane, typename Vec4<TIn>::T (&raw)[kBC]) {
    const TIn* base = x + (t0 * H + h) * kDim + 4 * lane;
    const int64_t stride = (int64_t)H * kDim;
#pragma unroll
    for (int i = 0; i < kBC; ++i)
        raw[i] = *reinterpret_cast<const typename Vec4<TIn>::T*>(base + (i < nt ? i : nt - 1) * stride);
}
__device__ __forceinline__ float4 ld4(const float* s, int r, int c) {
    return *reinterpret_cast<const float4*>(s + swz(r, c));
}
__device__ __forceinline__ void st4(float* s, int r, int c, float4 v) {
    *reinterpret_cast<float4*>(s + swz(r, c)) = v;
}
__device__ __forceinline__ float4 tf32r4(float4 v) {
    return make_float4(tf32r(v.x), tf32r(v.y), tf32r(v.z), tf32r(v.w));
}
__device__ __forceinline__ float4 zero_if(bool z, float4 v) {
    return z ? make_float4(0.f, 0.f, 0.f, 0.f) : v;
}

// Sequence of global chunk gc: the largest n < N with idx[n] <= gc.
__device__ __forceinline__ int find_seq(const int32_t* idx, int N, int64_t gc) {
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (idx[mid] <= gc) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(1024) kda_bwd_index_kernel(const int32_t* __restrict__ cu,
                                                             int N, int64_t host_chunks,
                                                             int64_t total_tokens,
                                                             int32_t* __restrict__ idx,
                                                             int* status) {
    __shared__ long long s_warp[32];
    __shared__ long long s_carry;
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        s_bad = cu[0] < 0;
        idx[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        long long c = 0;
        if (n < N) {
            const long long a = cu[n], b = cu[n + 1];
            if (b < a || b > total_tokens) s_bad = 1;
            else c = (b - a + kBC - 1) / kBC;
        }
        long long x = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            long long w = s_warp[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const long long incl = s_carry + x + (warp > 0 ? s_warp[warp - 1] : 0);
        if (n < N) idx[n + 1] = (int32_t)(incl > 0x7fffffffLL ? 0x7fffffff : incl);
        __syncthreads();
        if (tid == 1023) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) {
        const int stop = s_bad || s_carry != host_chunks;
        idx[N + 1] = stop;
        if (stop) report_status(status, KDA_ERR_INVALID_ARG);
    }
}

// TMA maps over the inputs, [T][H][128] (innermost first), box 128 channels x 1 head x 16 tokens:
// g, k, q, v of the input dtype and the fp32 output gradient.
struct BwdMaps {
    CUtensorMap g, k, q, v, d;
};

template <typename TIn>
struct BwdArgs {
    const TIn *q, *k, *v, *g, *beta;
    const int32_t* cu;
    const float* init_state;  // [N][H][128][128] or null
    const float* d_out;       // [T][H][128]
    const float* d_state;     // [N][H][128][128] or null
    float *dq, *dk, *dv, *dg, *dbeta, *d_init;
    const int32_t* idx;       // [N + 2]
    float* tiles;             // [chunks][H][3][16][16]: T, P, At
    float* states;            // [chunks][H][kSlot]: S^T at each chunk's start, then R = V - K_f S
    int* status;
    int N, H;
};

// At, P and T of one chunk of one head.
template <typename TIn>
__global__ void __launch_bounds__(kPrepThreads) kda_bwd_prep_kernel(const BwdArgs<TIn> p) {
    __shared__ __align__(16) float s_kp[kTile], s_km[kTile], s_qr[kTile];
    __shared__ float s_at[kBC][kBC + 1];
    __shared__ float s_beta[kBC];
    if (p.idx[p.N + 1]) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t gc = blockIdx.x;
    const int h = blockIdx.y, H = p.H;
    const int n = find_seq(p.idx, p.N, gc);
    const int64_t t0 = p.cu[n] + (gc - p.idx[n]) * kBC;
    const int nt = (int)(p.cu[n + 1] - t0 < kBC ? p.cu[n + 1] - t0 : kBC);
    {
        const int c = tid;  // key channel
        float G[kBC], kk[kBC], qq[kBC];
        load_col(p.g, t0, nt, H, h, c, G);
        load_col(p.k, t0, nt, H, h, c, kk);
        load_col(p.q, t0, nt, H, h, c, qq);
#pragma unroll
        for (int i = 1; i < kBC; ++i) G[i] += G[i - 1];
        const float r = 0.5f * G[kBC - 1];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < kBC; ++i) {
            const float x = G[i] - r;
            bad |= !(fabsf(x) <= kMaxExponent);
            const float ep = __expf(x), em = __expf(-x);
            s_kp[swz(i, c)] = tf32r(kk[i] * ep);
            s_km[swz(i, c)] = tf32r(kk[i] * em);
            s_qr[swz(i, c)] = tf32r(qq[i] * ep);
        }
        if (bad) report_status(p.status, kStatusDecayRange);
        if (tid < kBC) s_beta[tid] = tid < nt ? io<TIn>::to_f(p.beta[(t0 + tid) * H + h]) : 0.f;
    }
    __syncthreads();
    float* out = p.tiles + (gc * H + h) * (3 * kBC * kBC);
    {
        // warps 0, 1: At columns 0-7, 8-15; warps 2, 3: P columns 0-7, 8-15
        const int g = lane >> 2, t = lane & 3;
        const float* A = warp < 2 ? s_kp : s_qr;
        const int n0 = (warp & 1) * 8;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < kDim / 8; ++kk) {
            uint32_t a[4], b[2];
            lda_mk(A, 0, 8 * kk, g, t, a);
            ldb_nk(s_km, n0, 8 * kk, g, t, b);
            mma8(d, a, b);
        }
        const bool strict = warp < 2;
        float* o = out + (warp < 2 ? 2 : 1) * kBC * kBC;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = g + (e >> 1) * 8, col = n0 + 2 * t + (e & 1);
            const float x = (strict ? col < row : col <= row) ? d[e] : 0.f;
            o[row * kBC + col] = x;
            if (strict) s_at[row][col] = x;
        }
    }
    __syncthreads();
    if (warp == 0 && lane < kBC) {
        // column j of (I + diag(beta) At)^-1 by forward substitution
        const int j = lane;
        float x[kBC];
#pragma unroll
        for (int i = 0; i < kBC; ++i) {
            float acc = i == j ? 1.f : 0.f;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) s = fmaf(s_at[i][m], x[m], s);
            x[i] = acc - s_beta[i] * s;
        }
#pragma unroll
        for (int i = 0; i < kBC; ++i) out[i * kBC + j] = x[i];
    }
}

// Shared memory of the forward kernel, in floats.
struct FwdSmem {
    static constexpr int RAW = 0;                  // next chunk's g, k, v TMA boxes as loaded
    static constexpr int kRawTile = kTile;         // floats per box (fp32 inputs; bf16 use half)
    static constexpr int RAWT = RAW + 3 * kRawTile;  // next chunk's T tile
    static constexpr int KF = RAWT + kBC * kBC;    // K_f   [token][key]
    static constexpr int KBAR = KF + kTile;        // K_bar [token][key]
    static constexpr int V = KBAR + kTile;         // V     [token][value]
    static constexpr int GG = V + kTile;           // G     [token][key]
    static constexpr int KRAW = GG + kTile;        // k     [token][key]
    static constexpr int ST = KRAW + kTile;        // S^T being stored (swizzled tile)
    static constexpr int TB = ST + kState;         // T diag(beta)
    static constexpr int T = TB + kSmall;          // T
    static constexpr int A = T + kSmall;           // exp(G_C) per key
    static constexpr int BETA = A + kDim;
    static constexpr int BAR = BETA + kBC;         // mbarrier of the input copies
    static constexpr int RT = (BAR + 2 + 31) / 32 * 32;  // R of the last two chunks (swizzled)
    static constexpr int TOTAL = RT + 2 * kTile;
};
constexpr size_t kFwdSmemBytes = FwdSmem::TOTAL * sizeof(float);

// The forward state chain of one unit: S^T in registers, the start state of every chunk stored.
// Each chunk's inputs are loaded during the previous chunk.  The state, rounded to tf32 (it is
// only an MMA operand and a factor of one row sum later), leaves through a swizzled shared tile by
// one 64 KiB bulk asynchronous copy: the workspace holds that tile's image, which the reverse
// kernel copies back unchanged.  R = V - K_f S, which the reverse pass needs as it is, leaves the
// same way one chunk later (two tiles alternate).
template <typename TIn>
__global__ void __launch_bounds__(kBwdChainThreads, 1)
kda_bwd_forward_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs<TIn> p) {
    extern __shared__ __align__(128) float smf[];
    float* s_kf = smf + FwdSmem::KF;
    float* s_kbar = smf + FwdSmem::KBAR;
    float* s_v = smf + FwdSmem::V;
    float* s_tb = smf + FwdSmem::TB;
    float* s_a = smf + FwdSmem::A;
    float* s_st = smf + FwdSmem::ST;
    float* s_rt = smf + FwdSmem::RT;
    if (p.idx[p.N + 1]) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int H = p.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    const int64_t tb = p.cu[n], te = p.cu[n + 1];
    const int64_t c0 = p.idx[n];
    const int nch = p.idx[n + 1] - p.idx[n];
    const int dv0 = 16 * warp;  // value channels of this warp
    // S^T (value rows dv0.., key columns) as 16 accumulator tiles of 16 x 8
    float S[kDim / 8][4];
    {
        const float* s0 = p.init_state ? p.init_state + ((int64_t)n * H + h) * kState : nullptr;
#pragma unroll
        for (int j = 0; j < kDim / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = dv0 + g + (e >> 1) * 8, col = 8 * j + 2 * t + (e & 1);
                S[j][e] = s0 ? s0[col * kDim + row] : 0.f;
            }
    }
    // the next chunk's inputs, copied a chunk ahead: one TMA box each of g, k and v and a bulk
    // copy of the tile T, issued by thread 0 and completing on an mbarrier; beta by warp 3 into
    // registers
    float* s_G = smf + FwdSmem::GG;
    float* s_K = smf + FwdSmem::KRAW;
    float* s_T = smf + FwdSmem::T;
    float* s_beta = smf + FwdSmem::BETA;
    const TIn* raw = reinterpret_cast<const TIn*>(smf + FwdSmem::RAW);
    constexpr int kBoxElems = FwdSmem::kRawTile * 4 / (int)sizeof(TIn);   // box stride, elements
    const float* rawT = smf + FwdSmem::RAWT;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smf + FwdSmem::BAR);
    uint32_t phase = 0;
    if (tid == 0) {
        sm100::mbar_init(bar, 1);
        sm100::mbar_init_fence();
    }
    __syncthreads();
    float rbeta = 0.f;
    auto issue_inputs = [&](int c) {
        const int64_t t0 = tb + (int64_t)c * kBC;
        const int nt = (int)(te - t0 < kBC ? te - t0 : kBC);
        if (tid == 0) {
            sm100::mbar_arrive_expect_tx(bar, 3 * kBC * kDim * (int)sizeof(TIn) + kBC * kBC * 4);
            const CUtensorMap* m3[3] = {&maps.g, &maps.k, &maps.v};
#pragma unroll
            for (int m = 0; m < 3; ++m)
                sm100::tma_load_3d(const_cast<TIn*>(raw) + m * kBoxElems, m3[m], bar, 0, h, (int)t0);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                "%2, [%3];" ::"r"(smem_u32(rawT)),
                "l"(p.tiles + ((c0 + c) * H + h) * (3 * kBC * kBC)), "n"(kBC * kBC * 4),
                "r"(smem_u32(bar))
                : "memory");
        }
        if (warp == 3) rbeta = lane < nt && lane < kBC ? io<TIn>::to_f(p.beta[(t0 + lane) * H + h]) : 0.f;
    };
    if (nch > 0) issue_inputs(0);
    for (int c = 0; c < nch; ++c) {
        const int64_t slot = (c0 + c) * H + h;
        const int64_t t0 = tb + (int64_t)c * kBC;
        const int nt = (int)(te - t0 < kBC ? te - t0 : kBC);
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        // the chunk's inputs; a wait that gives up stops the unit (status KDA_ERR_TIMEOUT)
        const bool arrived = sm100::mbar_wait(bar, phase, kBwdWaitLimit);
        phase ^= 1u;
        if (__syncthreads_or(!arrived)) {
            if (tid == 0) {
                report_status(p.status, kStatusTimeout);
                sm100::mbar_wait(bar, phase ^ 1u, kBwdWaitLimit);
                asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            }
            return;
        }
        if (warp < 3) {
            // channels 4 lane .. 4 lane + 3 of the chunk's rows of g (warp 0), k (1) or v (2)
            const TIn* src = raw + warp * kBoxElems + 4 * lane;
            float4 G = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kBC; ++i) {
                const float4 x = zero_if(i >= nt, Vec4<TIn>::unpack(
                    *reinterpret_cast<const typename Vec4<TIn>::T*>(src + i * kDim)));
                if (warp == 0) {
                    G.x += x.x; G.y += x.y; G.z += x.z; G.w += x.w;
                    st4(s_G, i, 4 * lane, G);
                } else {
                    st4(warp == 1 ? s_K : s_v, i, 4 * lane, x);
                }
            }
            if (warp == 0)
                *reinterpret_cast<float4*>(s_a + 4 * lane) =
                    make_float4(__expf(G.x), __expf(G.y), __expf(G.z), __expf(G.w));
        } else if (warp == 3) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int e = 4 * lane + 128 * m;
                *reinterpret_cast<float4*>(s_T + (e >> 4) * kSmallLd + (e & 15)) =
                    *reinterpret_cast<const float4*>(rawT + e);
            }
            if (lane < kBC) s_beta[lane] = rbeta;
        }
        // the chunk's start state S^T [value][key] into the store tile
#pragma unroll
        for (int j = 0; j < kDim / 8; ++j) {
            const float st[4] = {tf32r(S[j][0]), tf32r(S[j][1]), tf32r(S[j][2]), tf32r(S[j][3])};
            st_c(s_st, dv0, 8 * j, g, t, st);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            asm volatile(
                "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                    p.states + slot * kSlot),
                "r"(smem_u32(s_st)), "n"(kState * 4)
                : "memory");
            if (c > 0)   // the previous chunk's R
                asm volatile(
                    "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                        p.states + (slot - H) * kSlot + kState),
                    "r"(smem_u32(s_rt + ((c - 1) & 1) * kTile)), "n"(kTile * 4)
                    : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        {
            // K_f = k e^G, K_bar = k e^(G_C - G): row tid >> 4, channels 4 (tid & 15) + 64 m
            const int i = tid >> 4;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int cb = 4 * (tid & 15) + 64 * m;
                const float4 G = ld4(s_G, i, cb), k4 = ld4(s_K, i, cb);
                const float4 GC = ld4(s_G, kBC - 1, cb);
                st4(s_kf, i, cb, tf32r4(make_float4(k4.x * __expf(G.x), k4.y * __expf(G.y),
                                                    k4.z * __expf(G.z), k4.w * __expf(G.w))));
                st4(s_kbar, i, cb, tf32r4(make_float4(k4.x * __expf(GC.x - G.x), k4.y * __expf(GC.y - G.y),
                                                      k4.z * __expf(GC.z - G.z), k4.w * __expf(GC.w - G.w))));
            }
            const int sc = tid & 15;
            s_tb[i * kSmallLd + sc] = tf32r(s_T[i * kSmallLd + sc] * s_beta[sc]);
        }
        __syncthreads();
        if (c + 1 < nch) issue_inputs(c + 1);
        // R^T = V^T - S^T K_f^T   (value rows, token columns)
        float R[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                R[jj][e] = s_v[swz(8 * jj + 2 * t + (e & 1), dv0 + g + (e >> 1) * 8)];
#pragma unroll
        for (int kk = 0; kk < kDim / 8; ++kk) {
            const uint32_t a[4] = {neg(tf32_bits(S[kk][0])), neg(tf32_bits(S[kk][2])),
                                   neg(tf32_bits(S[kk][1])), neg(tf32_bits(S[kk][3]))};
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                uint32_t b[2];
                ldb_nk(s_kf, 8 * jj, 8 * kk, g, t, b);
                mma8(R[jj], a, b);
            }
        }
        // R [token][value] into this chunk's R tile, for the reverse pass
        {
            float* rt = s_rt + (c & 1) * kTile;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    rt[swz(8 * jj + 2 * t + (e & 1), dv0 + g + (e >> 1) * 8)] = R[jj][e];
        }
        // U^T = R^T (T diag(beta))^T
        float U[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t a[4] = {tf32_bits(R[kk][0]), tf32_bits(R[kk][2]), tf32_bits(R[kk][1]),
                                   tf32_bits(R[kk][3])};
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const float2 v = *reinterpret_cast<const float2*>(
                    s_tb + (8 * jj + g) * kSmallLd + 8 * kk + 2 * t);
                const uint32_t b[2] = {bits(v.x), bits(v.y)};
                mma8(U[jj], a, b);
            }
        }
        // S^T <- S^T diag(a) + U^T K_bar
#pragma unroll
        for (int j = 0; j < kDim / 8; ++j) {
            const float a0 = s_a[8 * j + 2 * t], a1 = s_a[8 * j + 2 * t + 1];
            S[j][0] *= a0; S[j][1] *= a1; S[j][2] *= a0; S[j][3] *= a1;
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t a[4] = {tf32_bits(U[kk][0]), tf32_bits(U[kk][2]), tf32_bits(U[kk][1]),
                                   tf32_bits(U[kk][3])};
#pragma unroll
            for (int j = 0; j < kDim / 8; ++j) {
                uint32_t b[2];
                ldb_kn(s_kbar, 8 * kk, 8 * j, g, t, b);
                mma8(S[j], a, b);
            }
        }
    }
    // the last chunk's R, then every store must have completed before the CTA's shared memory is
    // released
    if (nch > 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0)
            asm volatile(
                "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
                "cp.async.bulk.commit_group;" ::"l"(p.states + ((c0 + nch - 1) * H + h) * kSlot + kState),
                "r"(smem_u32(s_rt + ((nch - 1) & 1) * kTile)), "n"(kTile * 4)
                : "memory");
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shared memory of the reverse kernel, in floats.
struct RevSmem {
    static constexpr int E = 0;                       // dE^T [value][key]
    static constexpr int KF = E + kState;             // K_f      [token][key]
    static constexpr int KBAR = KF + kTile;           // K_bar    [token][key]
    static constexpr int UU = KBAR + kTile;           // U        [token][value]
    static constexpr int RAW = KF;                    // bf16 inputs: K_f, K_bar, U hold the next
                                                      // chunk's boxes of g, k, q, v, dO as loaded
    static constexpr int QF = UU + kTile;             // Q_f      [token][key]
    static constexpr int W = QF + kTile;              // W        [token][key]
    static constexpr int KRAW = W + kTile;            // k        [token][key]
    static constexpr int QRAW = KRAW + kTile;         // q        [token][key]
    static constexpr int GG = QRAW + kTile;           // G        [token][key]
    static constexpr int DO = GG + kTile;             // dO       [token][value]
    static constexpr int RY = DO + kTile;             // V, R, then dY, then dG [token][value|key]
    static constexpr int DU = RY + kTile;             // dU       [token][value]
    static constexpr int T = DU + kTile;              // 16 x 16 tiles
    static constexpr int P = T + kSmall;
    static constexpr int AT = P + kSmall;
    static constexpr int TB = AT + kSmall;
    static constexpr int DA = TB + kSmall;
    static constexpr int DP = DA + kSmall;
    static constexpr int A = DP + kSmall;             // exp(G_C) per key
    static constexpr int R = A + kDim;                // G_C / 2 per key
    static constexpr int ES = R + kDim;               // rowsum(dE * S) per key
    static constexpr int CX = ES + kDim;              // sum_t dK_bar K_bar per key
    static constexpr int BETA = CX + kDim;
    static constexpr int DBP = BETA + kBC;            // per-warp partial rowsum(dY * R)
    static constexpr int SS = DBP + 8 * kBC;          // S^T [value][key] of the chunk (swizzled)
    static constexpr int BAR = SS + kState;           // mbarrier of the state's bulk copy
    static constexpr int BAR_IN = BAR + 2;            // mbarrier of the inputs' copies
    static constexpr int TOTAL = BAR_IN + 2;
};
constexpr size_t kRevSmemBytes = RevSmem::TOTAL * sizeof(float);

// The reverse pass of one unit: chunks from last to first, with dE^T (the gradient of the state at
// the end of the current chunk) in shared memory.
template <typename TIn>
__global__ void __launch_bounds__(kBwdChainThreads, 1)
kda_bwd_reverse_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs<TIn> p) {
    extern __shared__ __align__(128) float sm[];
    float* sE = sm + RevSmem::E;
    float* sKf = sm + RevSmem::KF;
    float* sKbar = sm + RevSmem::KBAR;
    float* sQf = sm + RevSmem::QF;
    float* sW = sm + RevSmem::W;
    float* sK = sm + RevSmem::KRAW;
    float* sQ = sm + RevSmem::QRAW;
    float* sG = sm + RevSmem::GG;
    float* sDO = sm + RevSmem::DO;
    float* sRY = sm + RevSmem::RY;
    float* sU = sm + RevSmem::UU;
    float* sDU = sm + RevSmem::DU;
    float* sT = sm + RevSmem::T;
    float* sP = sm + RevSmem::P;
    float* sAt = sm + RevSmem::AT;
    float* sTB = sm + RevSmem::TB;
    float* sDA = sm + RevSmem::DA;
    float* sDP = sm + RevSmem::DP;
    float* sA = sm + RevSmem::A;
    float* sR = sm + RevSmem::R;
    float* sES = sm + RevSmem::ES;
    float* sCX = sm + RevSmem::CX;
    float* sBeta = sm + RevSmem::BETA;
    float* sDBP = sm + RevSmem::DBP;

    if (p.idx[p.N + 1]) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int H = p.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    const int64_t tb = p.cu[n], te = p.cu[n + 1];
    const int64_t c0 = p.idx[n];
    const int nch = p.idx[n + 1] - p.idx[n];
    const int64_t ubase = ((int64_t)n * H + h) * kState;
    const int w16 = 16 * warp;  // this warp's value channels (phases 2, 4a) or key channels (3, 4b)

    // dE^T from the final-state gradient (or zero)
    for (int e = tid; e < kState; e += kBwdChainThreads) {
        const int dv = e & (kDim - 1), dk = e >> 7;   // read d_state[dk][dv] coalesced
        sE[swz(dv, dk)] = p.d_state ? p.d_state[ubase + e] : 0.f;
    }

    // the chunk's start state S^T and its R = V - K_f S (the forward kernel's swizzled tile
    // images) into shared memory, two bulk copies completing on an mbarrier; R lands in sRY, free
    // from phase 3 on (the chunk's dG goes to sDU)
    float* sS = sm + RevSmem::SS;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + RevSmem::BAR);
    uint32_t phase = 0;
    if (tid == 0) {
        sm100::mbar_init(bar, 1);
        sm100::mbar_init_fence();
    }
    __syncthreads();
    auto issue_state = [&](int c) {
        if (tid == 0) {
            const float* src = p.states + ((c0 + c) * H + h) * kSlot;
            sm100::mbar_arrive_expect_tx(bar, kSlot * 4);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
                "[%3];" ::"r"(smem_u32(sS)),
                "l"(src), "n"(kState * 4), "r"(smem_u32(bar))
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
                "[%3];" ::"r"(smem_u32(sRY)),
                "l"(src + kState), "n"(kTile * 4), "r"(smem_u32(bar))
                : "memory");
        }
    };
    // The next chunk's inputs, fetched a chunk ahead (v is not needed: R comes with the state).
    // bf16 inputs: one TMA box each of g, k, q and dO into the K_f / K_bar / U region (free from
    // phase 3 to the next staging), issued by thread 0 on the mbarrier bar_in.  fp32 inputs
    // (boxes twice as large): warps 0-2 load g, k, q and warps 4, 5 dO into registers (lane l:
    // channels 4l..4l+3).  Warp 6 loads the tiles T, P, At (six float4 a lane) and warp 7 beta.
    constexpr bool kBulkIn = sizeof(TIn) == 2;
    const TIn* rawIn = reinterpret_cast<const TIn*>(sm + RevSmem::RAW);   // [3][16][128]
    const float* rawDO = sm + RevSmem::RAW + 3 * kTile * (int)sizeof(TIn) / 4;  // [16][128]
    uint64_t* bar_in = reinterpret_cast<uint64_t*>(sm + RevSmem::BAR_IN);
    uint32_t phase_in = 0;
    if (tid == 0) {
        sm100::mbar_init(bar_in, 1);
        sm100::mbar_init_fence();
    }
    __syncthreads();
    using V4 = typename Vec4<TIn>::T;
    V4 rin[kBulkIn ? 1 : kBC];
    float4 rf[8];
    float rbeta = 0.f;
    auto issue_inputs = [&](int c) {
        const int64_t t0 = tb + (int64_t)c * kBC;
        const int nt = (int)(te - t0 < kBC ? te - t0 : kBC);
        if constexpr (kBulkIn) {
            if (tid == 0) {
                sm100::mbar_arrive_expect_tx(bar_in, 3 * kTile * (int)sizeof(TIn) + kTile * 4);
                const CUtensorMap* m4[3] = {&maps.g, &maps.k, &maps.q};
#pragma unroll
                for (int m = 0; m < 3; ++m)
                    sm100::tma_load_3d(const_cast<TIn*>(rawIn) + m * kTile, m4[m], bar_in, 0, h,
                                       (int)t0);
                sm100::tma_load_3d(const_cast<float*>(rawDO), &maps.d, bar_in, 0, h, (int)t0);
            }
        } else {
            if (warp < 3) {
                load_rows4(warp == 0 ? p.g : warp == 1 ? p.k : p.q, t0, nt, H, h, lane, rin);
            } else if (warp == 4 || warp == 5) {
                const float* base = p.d_out + (t0 * H + h) * kDim + 4 * lane;
                const int64_t stride = (int64_t)H * kDim;
                const int r0 = (warp - 4) * 8;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = r0 + i;
                    rf[i] = *reinterpret_cast<const float4*>(base + (row < nt ? row : nt - 1) * stride);
                }
            }
        }
        if (warp == 6) {
            const float* tl = p.tiles + ((c0 + c) * H + h) * (3 * kBC * kBC);
#pragma unroll
            for (int m = 0; m < 6; ++m)
                rf[m] = *reinterpret_cast<const float4*>(tl + 4 * (lane + 32 * m));
        } else if (warp == 7) {
            rbeta = lane < nt && lane < kBC ? io<TIn>::to_f(p.beta[(t0 + lane) * H + h]) : 0.f;
        }
    };
    // row i, channels 4 lane .. 4 lane + 3 of input m (0 g, 1 k, 2 q) and of dO
    auto in_row = [&](int m, int i) -> float4 {
        if constexpr (kBulkIn)
            return Vec4<TIn>::unpack(*reinterpret_cast<const V4*>(rawIn + m * kTile + i * kDim + 4 * lane));
        else
            return Vec4<TIn>::unpack(rin[i]);
    };
    auto do_row = [&](int i) -> float4 {
        if constexpr (kBulkIn)
            return *reinterpret_cast<const float4*>(rawDO + i * kDim + 4 * lane);
        else
            return rf[i & 7];
    };
    if (nch > 0) {
        issue_state(nch - 1);
        issue_inputs(nch - 1);
    }

    for (int c = nch - 1; c >= 0; --c) {
        const int64_t t0 = tb + (int64_t)c * kBC;
        const int nt = (int)(te - t0 < kBC ? te - t0 : kBC);
        {
            // the chunk's input copies; a wait that gives up stops the unit (KDA_ERR_TIMEOUT)
            const bool arrived = !kBulkIn || sm100::mbar_wait(bar_in, phase_in, kBwdWaitLimit);
            phase_in ^= 1u;
            if (__syncthreads_or(!arrived)) {
                if (tid == 0) {
                    report_status(p.status, kStatusTimeout);
                    sm100::mbar_wait(bar_in, phase_in ^ 1u, kBwdWaitLimit);
                    sm100::mbar_wait(bar, phase, kBwdWaitLimit);
                }
                return;
            }
        }
        // ---- phase 1: stage the chunk: warp 0 the prefix sums of g, warps 1, 2 k and q, warps
        // 4, 5 dO rows 0-7 and 8-15, warp 6 the tiles T, P, At, warp 7 beta ----
        if (warp == 0) {
            float4 G = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kBC; ++i) {
                const float4 x = zero_if(i >= nt, in_row(0, i));
                G.x += x.x; G.y += x.y; G.z += x.z; G.w += x.w;
                st4(sG, i, 4 * lane, G);
            }
            *reinterpret_cast<float4*>(sA + 4 * lane) =
                make_float4(__expf(G.x), __expf(G.y), __expf(G.z), __expf(G.w));
            *reinterpret_cast<float4*>(sR + 4 * lane) =
                make_float4(0.5f * G.x, 0.5f * G.y, 0.5f * G.z, 0.5f * G.w);
        } else if (warp < 3) {
            float* dst = warp == 1 ? sK : sQ;
#pragma unroll
            for (int i = 0; i < kBC; ++i) st4(dst, i, 4 * lane, zero_if(i >= nt, in_row(warp, i)));
        } else if (warp == 4 || warp == 5) {
            const int r0 = (warp - 4) * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st4(sDO, r0 + i, 4 * lane, zero_if(r0 + i >= nt, tf32r4(do_row(r0 + i))));
        } else if (warp == 6) {
#pragma unroll
            for (int m = 0; m < 6; ++m) {
                const int e = 4 * (lane + 32 * m), tile = e >> 8, r = (e & 255) >> 4, cc = e & 15;
                float* dst = (tile == 0 ? sT : tile == 1 ? sP : sAt) + r * kSmallLd + cc;
                *reinterpret_cast<float4*>(dst) = tile == 2 ? rf[m] : tf32r4(rf[m]);
            }
        } else if (warp == 7 && lane < kBC) {
            sBeta[lane] = rbeta;
        }
        __syncthreads();
        {
            // K_f = k e^G, Q_f = q e^G, K_bar = k e^(G_C - G): row tid >> 4, channels
            // 4 (tid & 15) + 64 m; and T diag(beta)
            const int i = tid >> 4;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int cb = 4 * (tid & 15) + 64 * m;
                const float4 G = ld4(sG, i, cb), k4 = ld4(sK, i, cb), q4 = ld4(sQ, i, cb);
                const float4 GC = ld4(sG, kBC - 1, cb);
                const float4 eg = make_float4(__expf(G.x), __expf(G.y), __expf(G.z), __expf(G.w));
                st4(sKf, i, cb, tf32r4(make_float4(k4.x * eg.x, k4.y * eg.y, k4.z * eg.z, k4.w * eg.w)));
                st4(sQf, i, cb, tf32r4(make_float4(q4.x * eg.x, q4.y * eg.y, q4.z * eg.z, q4.w * eg.w)));
                st4(sKbar, i, cb, tf32r4(make_float4(k4.x * __expf(GC.x - G.x), k4.y * __expf(GC.y - G.y),
                                                     k4.z * __expf(GC.z - G.z), k4.w * __expf(GC.w - G.w))));
            }
            const int sc = tid & 15;
            sTB[i * kSmallLd + sc] = tf32r(sT[i * kSmallLd + sc] * sBeta[sc]);
        }
        // the state's copy; a wait that gives up stops the unit (status KDA_ERR_TIMEOUT)
        const bool arrived = sm100::mbar_wait(bar, phase, kBwdWaitLimit);
        phase ^= 1u;
        if (__syncthreads_or(!arrived)) {
            if (tid == 0) {
                report_status(p.status, kStatusTimeout);
                sm100::mbar_wait(bar, phase ^ 1u, kBwdWaitLimit);
            }
            return;
        }
        // ---- phase 2 (value channels w16.. of this warp) ----
        // R = V - K_f S (token rows, value columns) arrived from the forward pass in sRY
        float R[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const float2 lo = *reinterpret_cast<const float2*>(sRY + swz(g, w16 + 8 * jj + 2 * t));
            const float2 hi = *reinterpret_cast<const float2*>(sRY + swz(g + 8, w16 + 8 * jj + 2 * t));
            R[jj][0] = lo.x; R[jj][1] = lo.y; R[jj][2] = hi.x; R[jj][3] = hi.y;
        }
        // U = T diag(beta) R
        {
            float U[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                lda_small(sTB, 8 * kk, g, t, a);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t b[2] = {
                        tf32_bits(sRY[swz(8 * kk + 2 * t, w16 + 8 * jj + g)]),
                        tf32_bits(sRY[swz(8 * kk + 2 * t + 1, w16 + 8 * jj + g)])};
                    mma8(U[jj], a, b);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] = tf32r(U[jj][e]);
                st_c(sU, 0, w16 + 8 * jj, g, t, u);
            }
        }
        // dU = K_bar dE + P^T dO
        {
            float D[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < kDim / 8; ++kk) {
                uint32_t a[4];
                lda_mk(sKbar, 0, 8 * kk, g, t, a);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t b[2];
                    const float2 v = *reinterpret_cast<const float2*>(
                        sE + swz(w16 + 8 * jj + g, 8 * kk + 2 * t));
                    b[0] = tf32_bits(v.x); b[1] = tf32_bits(v.y);
                    mma8(D[jj], a, b);
                }
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                lda_small_tr(sP, 8 * kk, g, t, a);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t b[2];
                    ldb_kn(sDO, 8 * kk, w16 + 8 * jj, g, t, b);
                    mma8(D[jj], a, b);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] = tf32r(D[jj][e]);
                st_c(sDU, 0, w16 + 8 * jj, g, t, u);
            }
        }
        __syncwarp();
        // dY = T^T dU; dbeta partial; dv = diag(beta) dY
        {
            float Y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                lda_small_tr(sT, 8 * kk, g, t, a);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t b[2];
                    ldb_kn(sDU, 8 * kk, w16 + 8 * jj, g, t, b);
                    mma8(Y[jj], a, b);
                }
            }
            float pb0 = 0.f, pb1 = 0.f;   // rows g, g + 8
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                pb0 += Y[jj][0] * R[jj][0] + Y[jj][1] * R[jj][1];
                pb1 += Y[jj][2] * R[jj][2] + Y[jj][3] * R[jj][3];
            }
            pb0 += __shfl_xor_sync(0xffffffffu, pb0, 1);
            pb0 += __shfl_xor_sync(0xffffffffu, pb0, 2);
            pb1 += __shfl_xor_sync(0xffffffffu, pb1, 1);
            pb1 += __shfl_xor_sync(0xffffffffu, pb1, 2);
            if (t == 0) {
                sDBP[warp * kBC + g] = pb0;
                sDBP[warp * kBC + g + 8] = pb1;
            }
            const float b0 = sBeta[g], b1 = sBeta[g + 8];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int col = w16 + 8 * jj + 2 * t;
                if (g < nt)
                    *reinterpret_cast<float2*>(p.dv + ((t0 + g) * H + h) * kDim + col) =
                        make_float2(b0 * Y[jj][0], b0 * Y[jj][1]);
                if (g + 8 < nt)
                    *reinterpret_cast<float2*>(p.dv + ((t0 + g + 8) * H + h) * kDim + col) =
                        make_float2(b1 * Y[jj][2], b1 * Y[jj][3]);
            }
            __syncwarp();   // this warp's reads of R in sRY are done
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = tf32r(Y[jj][e]);
                st_c(sRY, 0, w16 + 8 * jj, g, t, y);
            }
        }
        // W = T diag(beta) K_f   (key columns w16..)
        {
            float Wd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                lda_small(sTB, 8 * kk, g, t, a);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t b[2];
                    ldb_kn(sKf, 8 * kk, w16 + 8 * jj, g, t, b);
                    mma8(Wd[jj], a, b);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] = tf32r(Wd[jj][e]);
                st_c(sW, 0, w16 + 8 * jj, g, t, u);
            }
        }
        __syncthreads();  // dY, U, dU, W of all warps in shared memory
        // ---- phase 3 (key channels w16.. of this warp) ----
        float YS[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float QS[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float KB[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            // S^T rows 8kk+2t, 8kk+2t+1 (value), columns w16 + 8jj + g (key)
            float es[2] = {0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < kDim / 8; ++kk) {
                float sv[2][2];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    sv[jj][0] = sS[swz(8 * kk + 2 * t, w16 + 8 * jj + g)];
                    sv[jj][1] = sS[swz(8 * kk + 2 * t + 1, w16 + 8 * jj + g)];
                }
                uint32_t ay[4], ao[4], au[4];
                lda_mk(sRY, 0, 8 * kk, g, t, ay);
                lda_mk(sDO, 0, 8 * kk, g, t, ao);
                lda_mk(sU, 0, 8 * kk, g, t, au);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t b[2] = {bits(sv[jj][0]), bits(sv[jj][1])};
                    mma8(YS[jj], ay, b);
                    mma8(QS[jj], ao, b);
                    const float e0 = sE[swz(8 * kk + 2 * t, w16 + 8 * jj + g)];
                    const float e1 = sE[swz(8 * kk + 2 * t + 1, w16 + 8 * jj + g)];
                    es[jj] = fmaf(e0, sv[jj][0], fmaf(e1, sv[jj][1], es[jj]));
                    const uint32_t be[2] = {tf32_bits(e0), tf32_bits(e1)};
                    mma8(KB[jj], au, be);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                es[jj] += __shfl_xor_sync(0xffffffffu, es[jj], 1);
                es[jj] += __shfl_xor_sync(0xffffffffu, es[jj], 2);
                if (t == 0) sES[w16 + 8 * jj + g] = es[jj];
            }
        }
        // dA = -strict_lower(dY U^T), dP = lower_incl(dO U^T)   (warps 0-3)
        if (warp < 4) {
            const float* A = warp < 2 ? sRY : sDO;
            const int n0 = (warp & 1) * 8;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < kDim / 8; ++kk) {
                uint32_t a[4], b[2];
                lda_mk(A, 0, 8 * kk, g, t, a);
                ldb_nk(sU, n0, 8 * kk, g, t, b);
                mma8(d, a, b);
            }
            float* o = warp < 2 ? sDA : sDP;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = g + (e >> 1) * 8, col = n0 + 2 * t + (e & 1);
                o[row * kSmallLd + col] =
                    warp < 2 ? (col < row ? -d[e] : 0.f) : (col <= row ? d[e] : 0.f);
            }
        }
        __syncthreads();  // dA, dP, ES complete; every read of the old dE and of S done
        if (c > 0) {
            issue_state(c - 1);
            issue_inputs(c - 1);
        }
        // ---- phase 4a: dE^T <- dE^T diag(a) + dO^T Q_f - dU^T W   (value rows w16..) ----
        {
            float E[kDim / 8][4];
#pragma unroll
            for (int j = 0; j < kDim / 8; ++j) {
                const float a0 = sA[8 * j + 2 * t], a1 = sA[8 * j + 2 * t + 1];
                const float2 lo = *reinterpret_cast<const float2*>(sE + swz(w16 + g, 8 * j + 2 * t));
                const float2 hi = *reinterpret_cast<const float2*>(sE + swz(w16 + g + 8, 8 * j + 2 * t));
                E[j][0] = lo.x * a0; E[j][1] = lo.y * a1; E[j][2] = hi.x * a0; E[j][3] = hi.y * a1;
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t ao[4], au[4];
                lda_km(sDO, w16, 8 * kk, g, t, ao);
                lda_km(sDU, w16, 8 * kk, g, t, au);
                au[0] = neg(au[0]); au[1] = neg(au[1]); au[2] = neg(au[2]); au[3] = neg(au[3]);
#pragma unroll
                for (int j = 0; j < kDim / 8; ++j) {
                    uint32_t bq[2], bw[2];
                    ldb_kn(sQf, 8 * kk, 8 * j, g, t, bq);
                    ldb_kn(sW, 8 * kk, 8 * j, g, t, bw);
                    mma8(E[j], ao, bq);
                    mma8(E[j], au, bw);
                }
            }
#pragma unroll
            for (int j = 0; j < kDim / 8; ++j) st_c(sE, w16, 8 * j, g, t, E[j]);
        }
        // ---- phase 4b: the chunk's gradients (key channels w16..) ----
        {
            float KP[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float KM[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float QR[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const float bg0 = sBeta[g], bg1 = sBeta[g + 8];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                // A operands: diag(beta) dA, dP (rows t, k = s) and their transposes (rows s, k = t)
                uint32_t ada[4], adp[4], adat[4], adpt[4];
                {
                    const float2 lo = *reinterpret_cast<const float2*>(sDA + g * kSmallLd + 8 * kk + 2 * t);
                    const float2 hi = *reinterpret_cast<const float2*>(sDA + (g + 8) * kSmallLd + 8 * kk + 2 * t);
                    ada[0] = tf32_bits(bg0 * lo.x); ada[1] = tf32_bits(bg1 * hi.x);
                    ada[2] = tf32_bits(bg0 * lo.y); ada[3] = tf32_bits(bg1 * hi.y);
                }
                {
                    const float2 lo = *reinterpret_cast<const float2*>(sDP + g * kSmallLd + 8 * kk + 2 * t);
                    const float2 hi = *reinterpret_cast<const float2*>(sDP + (g + 8) * kSmallLd + 8 * kk + 2 * t);
                    adp[0] = tf32_bits(lo.x); adp[1] = tf32_bits(hi.x);
                    adp[2] = tf32_bits(lo.y); adp[3] = tf32_bits(hi.y);
                }
                {
                    const int r0 = 8 * kk + 2 * t, r1 = r0 + 1;
                    const float b0 = sBeta[r0], b1 = sBeta[r1];
                    adat[0] = tf32_bits(b0 * sDA[r0 * kSmallLd + g]);
                    adat[1] = tf32_bits(b0 * sDA[r0 * kSmallLd + g + 8]);
                    adat[2] = tf32_bits(b1 * sDA[r1 * kSmallLd + g]);
                    adat[3] = tf32_bits(b1 * sDA[r1 * kSmallLd + g + 8]);
                    adpt[0] = tf32_bits(sDP[r0 * kSmallLd + g]);
                    adpt[1] = tf32_bits(sDP[r0 * kSmallLd + g + 8]);
                    adpt[2] = tf32_bits(sDP[r1 * kSmallLd + g]);
                    adpt[3] = tf32_bits(sDP[r1 * kSmallLd + g + 8]);
                }
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int col = w16 + 8 * jj + g;
                    const float rr = sR[col];
                    const int o0 = swz(8 * kk + 2 * t, col), o1 = swz(8 * kk + 2 * t + 1, col);
                    const float x0 = sG[o0] - rr, x1 = sG[o1] - rr;
                    const float k0 = sK[o0], k1 = sK[o1];
                    const float ep0 = __expf(x0), ep1 = __expf(x1), em0 = __expf(-x0), em1 = __expf(-x1);
                    const uint32_t bkm[2] = {tf32_bits(k0 * em0), tf32_bits(k1 * em1)};
                    const uint32_t bkp[2] = {tf32_bits(k0 * ep0), tf32_bits(k1 * ep1)};
                    const uint32_t bqr[2] = {tf32_bits(sQ[o0] * ep0), tf32_bits(sQ[o1] * ep1)};
                    mma8(KP[jj], ada, bkm);
                    mma8(QR[jj], adp, bkm);
                    mma8(KM[jj], adat, bkp);
                    mma8(KM[jj], adpt, bqr);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = g + (e >> 1) * 8, col = w16 + 8 * jj + 2 * t + (e & 1);
                    const int o = swz(row, col);
                    const float Gv = sG[o], kv = sK[o], qv = sQ[o];
                    const float rr = sR[col], GC = 2.f * rr;
                    const float eg = __expf(Gv), egr = __expf(Gv - rr), erg = __expf(rr - Gv),
                                ecg = __expf(GC - Gv);
                    const float dKf = -sBeta[row] * YS[jj][e];
                    const float kterm = dKf * eg + KP[jj][e] * egr - KM[jj][e] * erg - KB[jj][e] * ecg;
                    const float qterm = QS[jj][e] * eg + QR[jj][e] * egr;
                    const float dkv = dKf * eg + KP[jj][e] * egr + KM[jj][e] * erg + KB[jj][e] * ecg;
                    YS[jj][e] = kv * kterm + qv * qterm;   // dG
                    QS[jj][e] = qterm;                     // dq
                    KP[jj][e] = dkv;                       // dk
                    KB[jj][e] *= kv * ecg;                 // dK_bar * K_bar
                }
            }
            // sum over the chunk's tokens of dK_bar * K_bar, per key column
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                float s0 = KB[jj][0] + KB[jj][2], s1 = KB[jj][1] + KB[jj][3];   // columns 2t, 2t+1
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    s0 += __shfl_xor_sync(0xffffffffu, s0, off);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, off);
                }
                if (g == 0) {
                    sCX[w16 + 8 * jj + 2 * t] = s0;
                    sCX[w16 + 8 * jj + 2 * t + 1] = s1;
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int col = w16 + 8 * jj + 2 * t;
                if (g < nt) {
                    const int64_t o = ((t0 + g) * H + h) * kDim + col;
                    *reinterpret_cast<float2*>(p.dk + o) = make_float2(KP[jj][0], KP[jj][1]);
                    *reinterpret_cast<float2*>(p.dq + o) = make_float2(QS[jj][0], QS[jj][1]);
                }
                if (g + 8 < nt) {
                    const int64_t o = ((t0 + g + 8) * H + h) * kDim + col;
                    *reinterpret_cast<float2*>(p.dk + o) = make_float2(KP[jj][2], KP[jj][3]);
                    *reinterpret_cast<float2*>(p.dq + o) = make_float2(QS[jj][2], QS[jj][3]);
                }
                st_c(sDU, 0, w16 + 8 * jj, g, t, YS[jj]);   // dG, in this warp's own columns
            }
            __syncwarp();
            {
                // dg = suffix sum of dG over the chunk (the chunk end also carries the G_C terms):
                // lanes 16-31 sum rows 15..8 of column w16 + (lane & 15), lanes 0-15 rows 7..0 and
                // then add the upper half's total
                const int col = w16 + (lane & 15), hi = lane >> 4;
                float part[8];
                float acc = hi ? sCX[col] + sA[col] * sES[col] : 0.f;
#pragma unroll
                for (int j = 7; j >= 0; --j) {
                    acc += sDU[swz(8 * hi + j, col)];
                    part[j] = acc;
                }
                const float upper = __shfl_sync(0xffffffffu, acc, lane | 16);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = 8 * hi + j;
                    if (i < nt) p.dg[((t0 + i) * H + h) * kDim + col] = hi ? part[j] : part[j] + upper;
                }
            }
        }
        if (warp == 7 && lane < kBC && lane < nt) {
            const int i = lane;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += sDBP[w * kBC + i];
#pragma unroll
            for (int s = 0; s < kBC; ++s) acc = fmaf(sDA[i * kSmallLd + s], sAt[i * kSmallLd + s], acc);
            p.dbeta[(t0 + i) * H + h] = acc;
        }
    }
    __syncthreads();
    // the gradient of the initial state, [key][value]
    for (int e = tid; e < kState; e += kBwdChainThreads) {
        const int dv = e & (kDim - 1), dk = e >> 7;
        p.d_init[ubase + e] = sE[swz(dv, dk)];
    }
}

PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over [T, H, 128] (innermost first) of `esize`-byte elements, box 128 x 1 x 16, no
// swizzle (rows land dense in shared memory); rows past T read as zero.
bool make_box_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, size_t esize,
                  int64_t T, int H) {
    auto enc = bwd_encode_fn();
    if (!enc || !base) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kDim * esize, (cuuint64_t)H * kDim * esize};
    cuuint32_t box[3] = {(cuuint32_t)kDim, 1, (cuuint32_t)kBC};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

size_t backward_workspace_floats(int num_seqs, int heads, int64_t chunks) {
    const size_t idx_floats = ((size_t)num_seqs + 2 + 63) / 64 * 64;
    return idx_floats + (size_t)chunks * heads * (3 * kBC * kBC + kSlot);
}

int64_t backward_chunks(const int32_t* host_seqlens, int num_seqs) {
    int64_t c = 0;
    for (int n = 0; n < num_seqs; ++n) c += ((int64_t)host_seqlens[n] + kBC - 1) / kBC;
    return c;
}

cudaError_t launch_backward(int dtype, int num_seqs, int heads, const void* q, const void* k,
                            const void* v, const void* g, const void* beta,
                            const int32_t* cu_seqlens, const float* init_state,
                            const float* d_out, const float* d_state, float* dq, float* dk,
                            float* dv, float* dg, float* dbeta, float* d_init, float* work,
                            int64_t chunks, int64_t total_tokens, int* status,
                            cudaStream_t stream) {
    if ((int64_t)num_seqs * heads <= 0) return cudaSuccess;
    int32_t* idx = reinterpret_cast<int32_t*>(work);
    const size_t idx_floats = ((size_t)num_seqs + 2 + 63) / 64 * 64;
    float* tiles = work + idx_floats;
    float* states = tiles + (size_t)chunks * heads * (3 * kBC * kBC);
    kda_bwd_index_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, num_seqs, chunks, total_tokens, idx,
                                                 status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto run = [&](auto tag) -> cudaError_t {
        using T = decltype(tag);
        const BwdArgs<T> a{(const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta,
                           cu_seqlens, init_state, d_out, d_state, dq, dk, dv, dg, dbeta, d_init,
                           idx, tiles, states, status, num_seqs, heads};
        BwdMaps maps;
        memset(&maps, 0, sizeof(maps));
        const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        if (total_tokens > 0 &&
            !(make_box_map(&maps.g, g, dt, sizeof(T), total_tokens, heads) &&
              make_box_map(&maps.k, k, dt, sizeof(T), total_tokens, heads) &&
              make_box_map(&maps.q, q, dt, sizeof(T), total_tokens, heads) &&
              make_box_map(&maps.v, v, dt, sizeof(T), total_tokens, heads) &&
              make_box_map(&maps.d, d_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, total_tokens,
                           heads)))
            return cudaErrorInvalidValue;
        if (chunks > 0) {
            kda_bwd_prep_kernel<T><<<dim3((unsigned)chunks, (unsigned)heads), kPrepThreads, 0,
                                     stream>>>(a);
            cudaError_t err = cudaGetLastError();
            if (err != cudaSuccess) return err;
            err = cudaFuncSetAttribute(kda_bwd_forward_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kFwdSmemBytes);
            if (err != cudaSuccess) return err;
            kda_bwd_forward_kernel<T><<<(unsigned)(num_seqs * heads), kBwdChainThreads,
                                        kFwdSmemBytes, stream>>>(maps, a);
            err = cudaGetLastError();
            if (err != cudaSuccess) return err;
        }
        cudaError_t err = cudaFuncSetAttribute(kda_bwd_reverse_kernel<T>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kRevSmemBytes);
        if (err != cudaSuccess) return err;
        kda_bwd_reverse_kernel<T><<<(unsigned)(num_seqs * heads), kBwdChainThreads, kRevSmemBytes,
                                    stream>>>(maps, a);
        return cudaGetLastError();
    };
    if (dtype == KDA_BF16) return run(__nv_bfloat16{});
    return run(float{});
}

}  // namespace kda
