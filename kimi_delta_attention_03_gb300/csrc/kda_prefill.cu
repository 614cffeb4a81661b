// kda_prefill.cu — chunked KDA prefill over packed variable-length sequences.
//
// Method ("How Kimi K3 Engineered Its Way to the Frontier", section "FlashKDA steps the state
// once per 16 tokens"): split each sequence into fixed chunks, do the chunk-local work as
// dense tensor-core matmuls, and step the state once per chunk; the result equals the token
// loop.  This build uses 64-token chunks aligned to each sequence's own start; the last
// partial chunk is zero-padded (k = v = q = 0, beta = 0, g = 0), which adds nothing.
//
// Per chunk, with G the inclusive cumulative sum of g inside the chunk, G_C its last row and
// r = G_C / 2 a per-channel mid-chunk reference (it halves the exponent range of the
// reciprocal-decay rescaling, which the page notes can overflow in finite precision):
//   Q_r = q e^{G-r},  K_p = k e^{G-r},  K_m = k e^{r-G},  K_bar = k e^{G_C-G}
//   A   = strict_lower(diag(beta) K_p K_m^T)         P = lower_incl(Q_r K_m^T)
//   T   = (I + A)^{-1}                               (unit lower triangular, 64 x 64)
//   W   = T diag(beta) K_p                           U_bar = T diag(beta) V
//   S'  = diag(e^{r}) S   (bf16 operand copy of the fp32 state)
//   U   = U_bar - W S'      O = Q_r S' + P U      S <- diag(e^{G_C}) S + K_bar^T U
//
// Execution: one CTA per (sequence, head), 8 warps.  All products run on the tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate); the fp32 state stays in accumulator
// registers across chunks (warp w owns key channels 16w..16w+15, all 128 value channels).
// The 64 x 64 inverse is done in fp32 on the CUDA cores: 16 x 16 diagonal blocks by forward
// substitution (one column per thread), off-diagonal blocks by block forward substitution.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int LDK = 136;  // padded bf16 row for 128-wide tiles (272 B: conflict-free ldmatrix)
constexpr int LDC = 72;   // padded bf16 row for 64-wide tiles (144 B)
constexpr int LDA = 68;   // fp32 row of the 64 x 64 A / T matrix
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxExponent = 80.f;  // |G - r| bound; e^80 ~ 5.5e34 keeps bf16/fp32 finite

// shared-memory carve-up (bytes)
constexpr int kTile128 = kChunk * LDK * 2;       // 17408
constexpr int kOffQ = 0;                          // q, then Q_r in place
constexpr int kOffK = kOffQ + kTile128;           // raw k, later U
constexpr int kOffKp = kOffK + kTile128;          // K_p
constexpr int kOffKm = kOffKp + kTile128;         // K_m, later W
constexpr int kOffKb = kOffKm + kTile128;         // K_bar
constexpr int kOffV = kOffKb + kTile128;          // v
constexpr int kOffG = kOffV + kTile128;           // g fp32 [64][128], later A/T fp32 + Y
constexpr int kOffP = kOffG + kChunk * kDim * 4;  // P bf16 [64][LDC]
constexpr int kOffT = kOffP + kChunk * LDC * 2;   // T diag(beta) bf16 [64][LDC]
constexpr int kOffS = kOffT + kChunk * LDC * 2;   // S' bf16 [128][LDK]
constexpr int kOffBeta = kOffS + kDim * LDK * 2;  // fp32 [64]
constexpr int kOffPart = kOffBeta + kChunk * 4;   // fp32 [2][128]
constexpr int kOffEr = kOffPart + 2 * kDim * 4;   // fp32 [128]  e^{r}
constexpr int kOffGam = kOffEr + kDim * 4;        // fp32 [128]  e^{G_C}
constexpr int kSmemBytes = kOffGam + kDim * 4;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kChunk * LDA * 4 + 3 * 256 * 4 <= kChunk * kDim * 4, "A/T + Y fit the g region");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment (16 x 16, row-major source [M][K], leading dim ld elements) at (row0, col0).
__device__ __forceinline__ void load_a(const __nv_bfloat16* base, int ld, int row0, int col0,
                                       int lane, uint32_t (&a)[4]) {
    const __nv_bfloat16* p = base + (row0 + (lane & 15)) * ld + col0 + 8 * (lane >> 4);
    ldsm_x4(smem_u32(p), a);
}
// A fragment of X^T where X is stored [K][M] (rows = K): uses the transposing load.
__device__ __forceinline__ void load_a_trans(const __nv_bfloat16* base, int ld, int m0, int k0,
                                             int lane, uint32_t (&a)[4]) {
    const __nv_bfloat16* p =
        base + (k0 + (lane & 7) + 8 * (lane >> 4)) * ld + m0 + 8 * ((lane >> 3) & 1);
    ldsm_x4_t(smem_u32(p), a);
}
// B fragments of two adjacent n-tiles (n0, n0+8) for k-slice k0, source stored [N][K].
__device__ __forceinline__ void load_b_nk(const __nv_bfloat16* base, int ld, int n0, int k0,
                                          int lane, uint32_t (&b)[4]) {
    const __nv_bfloat16* p =
        base + (n0 + (lane & 7) + 8 * (lane >> 4)) * ld + k0 + 8 * ((lane >> 3) & 1);
    ldsm_x4(smem_u32(p), b);
}
// B fragments of two adjacent n-tiles (n0, n0+8) for k-slice k0, source stored [K][N].
__device__ __forceinline__ void load_b_kn(const __nv_bfloat16* base, int ld, int n0, int k0,
                                          int lane, uint32_t (&b)[4]) {
    const __nv_bfloat16* p =
        base + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ld + n0 + 8 * (lane >> 4);
    ldsm_x4_t(smem_u32(p), b);
}

__device__ __forceinline__ void store_bf16x2(__nv_bfloat16* base, int ld, int row, int col,
                                             float x, float y) {
    *reinterpret_cast<uint32_t*>(base + row * ld + col) = pack_bf16(x, y);
}

template <typename TIn> struct out_store;
template <> struct out_store<__nv_bfloat16> {
    static __device__ __forceinline__ void put(__nv_bfloat16* p, float x, float y) {
        *reinterpret_cast<uint32_t*>(p) = pack_bf16(x, y);
    }
};
template <> struct out_store<float> {
    static __device__ __forceinline__ void put(float* p, float x, float y) {
        *reinterpret_cast<float2*>(p) = make_float2(x, y);
    }
};

// Load one chunk of q, k, v (to bf16 tiles), g (to fp32) and beta; rows >= valid are zeros.
template <typename TIn>
__device__ __forceinline__ void load_chunk(unsigned char* smem, const TIn* q, const TIn* k,
                                           const TIn* v, const TIn* g, const TIn* beta,
                                           int64_t tok0, int valid, int H, int h, int tid) {
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + kOffQ);
    __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem + kOffK);
    __nv_bfloat16* sV = reinterpret_cast<__nv_bfloat16*>(smem + kOffV);
    float* sG = reinterpret_cast<float*>(smem + kOffG);
    float* sBeta = reinterpret_cast<float*>(smem + kOffBeta);
    const int64_t row_stride = (int64_t)H * kDim;
    if constexpr (sizeof(TIn) == 2) {
        // 16 vectors of 8 bf16 per row
        for (int e = tid; e < kChunk * 16; e += kThreads) {
            const int row = e >> 4, c8 = (e & 15) * 8;
            uint4 vq = make_uint4(0, 0, 0, 0), vk = vq, vv = vq, vg = vq;
            if (row < valid) {
                const int64_t off = (tok0 + row) * row_stride + (int64_t)h * kDim + c8;
                vq = *reinterpret_cast<const uint4*>(q + off);
                vk = *reinterpret_cast<const uint4*>(k + off);
                vv = *reinterpret_cast<const uint4*>(v + off);
                vg = *reinterpret_cast<const uint4*>(g + off);
            }
            *reinterpret_cast<uint4*>(sQ + row * LDK + c8) = vq;
            *reinterpret_cast<uint4*>(sK + row * LDK + c8) = vk;
            *reinterpret_cast<uint4*>(sV + row * LDK + c8) = vv;
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&vg);
            float4 lo, hi;
            float2 f0 = __bfloat1622float2(g2[0]), f1 = __bfloat1622float2(g2[1]);
            float2 f2 = __bfloat1622float2(g2[2]), f3 = __bfloat1622float2(g2[3]);
            lo = make_float4(f0.x, f0.y, f1.x, f1.y);
            hi = make_float4(f2.x, f2.y, f3.x, f3.y);
            *reinterpret_cast<float4*>(sG + row * kDim + c8) = lo;
            *reinterpret_cast<float4*>(sG + row * kDim + c8 + 4) = hi;
        }
    } else {
        // 32 vectors of 4 floats per row
        for (int e = tid; e < kChunk * 32; e += kThreads) {
            const int row = e >> 5, c4 = (e & 31) * 4;
            float4 vq = make_float4(0.f, 0.f, 0.f, 0.f), vk = vq, vv = vq, vg = vq;
            if (row < valid) {
                const int64_t off = (tok0 + row) * row_stride + (int64_t)h * kDim + c4;
                vq = *reinterpret_cast<const float4*>(q + off);
                vk = *reinterpret_cast<const float4*>(k + off);
                vv = *reinterpret_cast<const float4*>(v + off);
                vg = *reinterpret_cast<const float4*>(g + off);
            }
            uint2 pq = make_uint2(pack_bf16(vq.x, vq.y), pack_bf16(vq.z, vq.w));
            uint2 pk = make_uint2(pack_bf16(vk.x, vk.y), pack_bf16(vk.z, vk.w));
            uint2 pv = make_uint2(pack_bf16(vv.x, vv.y), pack_bf16(vv.z, vv.w));
            *reinterpret_cast<uint2*>(sQ + row * LDK + c4) = pq;
            *reinterpret_cast<uint2*>(sK + row * LDK + c4) = pk;
            *reinterpret_cast<uint2*>(sV + row * LDK + c4) = pv;
            *reinterpret_cast<float4*>(sG + row * kDim + c4) = vg;
        }
    }
    if (tid < kChunk)
        sBeta[tid] = tid < valid ? io<TIn>::to_f(beta[(tok0 + tid) * H + h]) : 0.f;
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                   const TIn* __restrict__ v, const TIn* __restrict__ g,
                   const TIn* __restrict__ beta, const float* __restrict__ init_state,
                   const int32_t* __restrict__ cu_seqlens, TIn* __restrict__ out,
                   float* __restrict__ final_state, int H, int* status) {
    extern __shared__ __align__(128) unsigned char smem[];
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + kOffQ);
    __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem + kOffK);
    __nv_bfloat16* sKp = reinterpret_cast<__nv_bfloat16*>(smem + kOffKp);
    __nv_bfloat16* sKm = reinterpret_cast<__nv_bfloat16*>(smem + kOffKm);
    __nv_bfloat16* sKb = reinterpret_cast<__nv_bfloat16*>(smem + kOffKb);
    __nv_bfloat16* sV = reinterpret_cast<__nv_bfloat16*>(smem + kOffV);
    float* sG = reinterpret_cast<float*>(smem + kOffG);
    float* sA = sG;                         // [64][LDA] after the factor pass
    float* sY = sG + kChunk * LDA;          // [3][16][16]
    __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(smem + kOffP);
    __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(smem + kOffT);
    __nv_bfloat16* sS = reinterpret_cast<__nv_bfloat16*>(smem + kOffS);
    float* sBeta = reinterpret_cast<float*>(smem + kOffBeta);
    float* sPart = reinterpret_cast<float*>(smem + kOffPart);
    float* sEr = reinterpret_cast<float*>(smem + kOffEr);
    float* sGam = reinterpret_cast<float*>(smem + kOffGam);

    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gq = lane >> 2;  // fragment row group
    const int tq = lane & 3;   // fragment column pair
    const int64_t seq0 = cu_seqlens[n];
    const int L = cu_seqlens[n + 1] - cu_seqlens[n];
    const int64_t unit = (int64_t)n * H + h;

    // fp32 state: rows 16*warp + gq (+8), columns 8*nt + 2*tq (+1)
    float Sf[16][4];
    {
        const int r0 = 16 * warp + gq;
        if (init_state) {
            const float* s0 = init_state + unit * (kDim * kDim);
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const float2 a = *reinterpret_cast<const float2*>(s0 + r0 * kDim + 8 * nt + 2 * tq);
                const float2 b = *reinterpret_cast<const float2*>(s0 + (r0 + 8) * kDim + 8 * nt + 2 * tq);
                Sf[nt][0] = a.x; Sf[nt][1] = a.y; Sf[nt][2] = b.x; Sf[nt][3] = b.y;
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) Sf[nt][0] = Sf[nt][1] = Sf[nt][2] = Sf[nt][3] = 0.f;
        }
    }

    for (int c0 = 0; c0 < L; c0 += kChunk) {
        const int valid = min(kChunk, L - c0);
        const int64_t tok0 = seq0 + c0;
        __syncthreads();  // previous chunk is done with every shared tile
        load_chunk<TIn>(smem, q, k, v, g, beta, tok0, valid, H, h, tid);
        __syncthreads();

        // ---- cumulative log-decay and the four rescaled tiles ----
        {
            const int c = tid & (kDim - 1);
            const int half = tid >> 7;
            float part = 0.f;
#pragma unroll 8
            for (int t = 32 * half; t < 32 * half + 32; ++t) part += sG[t * kDim + c];
            sPart[half * kDim + c] = part;
            __syncthreads();
            const float GC = sPart[c] + sPart[kDim + c];
            const float r = 0.5f * GC;
            float G = half ? sPart[c] : 0.f;
            bool bad = false;
            for (int t = 32 * half; t < 32 * half + 32; ++t) {
                G += sG[t * kDim + c];
                const float d = G - r;
                bad |= fabsf(d) > kMaxExponent;
                const float e = exp2f(d * kLog2e);
                const float ei = exp2f(-d * kLog2e);
                const float eb = exp2f((GC - G) * kLog2e);
                const float qv = __bfloat162float(sQ[t * LDK + c]);
                const float kv = __bfloat162float(sK[t * LDK + c]);
                sQ[t * LDK + c] = __float2bfloat16_rn(qv * e);
                sKp[t * LDK + c] = __float2bfloat16_rn(kv * e);
                sKm[t * LDK + c] = __float2bfloat16_rn(kv * ei);
                sKb[t * LDK + c] = __float2bfloat16_rn(kv * eb);
            }
            if (bad) report_status(status, kStatusDecayRange);
            if (half == 0) {
                sEr[c] = exp2f(r * kLog2e);
                sGam[c] = exp2f(GC * kLog2e);
            }
        }
        __syncthreads();

        // ---- S' = diag(e^r) S as the bf16 operand copy ----
        {
            const int r0 = 16 * warp + gq;
            const float e0 = sEr[r0], e1 = sEr[r0 + 8];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                store_bf16x2(sS, LDK, r0, 8 * nt + 2 * tq, Sf[nt][0] * e0, Sf[nt][1] * e0);
                store_bf16x2(sS, LDK, r0 + 8, 8 * nt + 2 * tq, Sf[nt][2] * e1, Sf[nt][3] * e1);
            }
        }

        // ---- A = strict_lower(beta K_p K_m^T) (warps 0-3), P = lower(Q_r K_m^T) (4-7) ----
        {
            const __nv_bfloat16* srcA = warp < 4 ? sKp : sQ;
            const int m0 = 16 * (warp & 3);
            float acc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                load_a(srcA, LDK, m0, 16 * ks, lane, a);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    load_b_nk(sKm, LDK, 16 * np, 16 * ks, lane, b);
                    mma16816(acc[2 * np], a, b[0], b[1]);
                    mma16816(acc[2 * np + 1], a, b[2], b[3]);
                }
            }
            const int i0 = m0 + gq, i1 = i0 + 8;
            if (warp < 4) {
                const float b0 = sBeta[i0], b1 = sBeta[i1];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int j = 8 * nt + 2 * tq;
                    float2 r0v = make_float2(j < i0 ? b0 * acc[nt][0] : 0.f,
                                             j + 1 < i0 ? b0 * acc[nt][1] : 0.f);
                    float2 r1v = make_float2(j < i1 ? b1 * acc[nt][2] : 0.f,
                                             j + 1 < i1 ? b1 * acc[nt][3] : 0.f);
                    *reinterpret_cast<float2*>(sA + i0 * LDA + j) = r0v;
                    *reinterpret_cast<float2*>(sA + i1 * LDA + j) = r1v;
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int j = 8 * nt + 2 * tq;
                    store_bf16x2(sP, LDC, i0, j, j <= i0 ? acc[nt][0] : 0.f,
                                 j + 1 <= i0 ? acc[nt][1] : 0.f);
                    store_bf16x2(sP, LDC, i1, j, j <= i1 ? acc[nt][2] : 0.f,
                                 j + 1 <= i1 ? acc[nt][3] : 0.f);
                }
            }
        }
        __syncthreads();

        // ---- T = (I + A)^{-1}: diagonal 16x16 blocks, one column per thread ----
        if (tid < 64) {
            const int b = tid >> 4, col = tid & 15;
            const float* Ab = sA + (16 * b) * LDA + 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = (i == col) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) s = fmaf(-Ab[i * LDA + j], x[j], s);
                x[i] = s;
            }
            __syncwarp();
            float* Tb = sA + (16 * b) * LDA + 16 * b;
#pragma unroll
            for (int i = 0; i < 16; ++i) Tb[i * LDA + col] = x[i];
        }
        __syncthreads();
        // ---- off-diagonal blocks: T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ ----
        for (int I = 1; I < 4; ++I) {
            for (int e = tid; e < I * 256; e += kThreads) {
                const int J = e >> 8, i = (e >> 4) & 15, j = e & 15;
                float y = 0.f;
                for (int K = J; K < I; ++K) {
                    const float* Arow = sA + (16 * I + i) * LDA + 16 * K;
                    const float* Tcol = sA + (16 * K) * LDA + 16 * J + j;
#pragma unroll
                    for (int x = 0; x < 16; ++x) y = fmaf(Arow[x], Tcol[x * LDA], y);
                }
                sY[e] = y;
            }
            __syncthreads();
            for (int e = tid; e < I * 256; e += kThreads) {
                const int J = e >> 8, i = (e >> 4) & 15, j = e & 15;
                const float* Trow = sA + (16 * I + i) * LDA + 16 * I;
                const float* Ycol = sY + J * 256 + j;
                float y = 0.f;
#pragma unroll
                for (int x = 0; x < 16; ++x) y = fmaf(Trow[x], Ycol[x * 16], y);
                sA[(16 * I + i) * LDA + 16 * J + j] = -y;
            }
            __syncthreads();
        }
        // ---- T diag(beta) as a bf16 operand ----
        for (int e = tid; e < kChunk * kChunk / 2; e += kThreads) {
            const int i = e >> 5, j = (e & 31) * 2;
            store_bf16x2(sT, LDC, i, j, sA[i * LDA + j] * sBeta[j],
                         sA[i * LDA + j + 1] * sBeta[j + 1]);
        }
        __syncthreads();

        // ---- W = T diag(beta) K_p (warps 0-3) and U_bar = T diag(beta) V (warps 4-7) ----
        float acc2[16][4];
        {
            const __nv_bfloat16* srcB = warp < 4 ? sKp : sV;
            const int m0 = 16 * (warp & 3);
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a(sT, LDC, m0, 16 * ks, lane, a);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b[4];
                    load_b_kn(srcB, LDK, 16 * np, 16 * ks, lane, b);
                    mma16816(acc2[2 * np], a, b[0], b[1]);
                    mma16816(acc2[2 * np + 1], a, b[2], b[3]);
                }
            }
            if (warp < 4) {
                const int i0 = m0 + gq;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    store_bf16x2(sKm, LDK, i0, 8 * nt + 2 * tq, acc2[nt][0], acc2[nt][1]);
                    store_bf16x2(sKm, LDK, i0 + 8, 8 * nt + 2 * tq, acc2[nt][2], acc2[nt][3]);
                }
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.f;
            } else {
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    acc2[nt][0] = -acc2[nt][0]; acc2[nt][1] = -acc2[nt][1];
                    acc2[nt][2] = -acc2[nt][2]; acc2[nt][3] = -acc2[nt][3];
                }
            }
        }
        __syncthreads();

        // ---- [Q_r ; W] S': warps 0-3 get Q_r S', warps 4-7 get W S' - U_bar = -U ----
        {
            const __nv_bfloat16* srcA = warp < 4 ? sQ : sKm;
            const int m0 = 16 * (warp & 3);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t a[4];
                load_a(srcA, LDK, m0, 16 * ks, lane, a);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b[4];
                    load_b_kn(sS, LDK, 16 * np, 16 * ks, lane, b);
                    mma16816(acc2[2 * np], a, b[0], b[1]);
                    mma16816(acc2[2 * np + 1], a, b[2], b[3]);
                }
            }
            if (warp >= 4) {
                const int i0 = m0 + gq;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    store_bf16x2(sK, LDK, i0, 8 * nt + 2 * tq, -acc2[nt][0], -acc2[nt][1]);
                    store_bf16x2(sK, LDK, i0 + 8, 8 * nt + 2 * tq, -acc2[nt][2], -acc2[nt][3]);
                }
            }
        }
        __syncthreads();

        // ---- O = Q_r S' + P U (warps 0-3), written to global for valid rows ----
        if (warp < 4) {
            const int m0 = 16 * warp;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a(sP, LDC, m0, 16 * ks, lane, a);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b[4];
                    load_b_kn(sK, LDK, 16 * np, 16 * ks, lane, b);
                    mma16816(acc2[2 * np], a, b[0], b[1]);
                    mma16816(acc2[2 * np + 1], a, b[2], b[3]);
                }
            }
            const int i0 = m0 + gq, i1 = i0 + 8;
            TIn* o0 = out + ((tok0 + i0) * H + h) * (int64_t)kDim;
            TIn* o1 = out + ((tok0 + i1) * H + h) * (int64_t)kDim;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int j = 8 * nt + 2 * tq;
                if (i0 < valid) out_store<TIn>::put(o0 + j, acc2[nt][0], acc2[nt][1]);
                if (i1 < valid) out_store<TIn>::put(o1 + j, acc2[nt][2], acc2[nt][3]);
            }
        }

        // ---- S <- diag(e^{G_C}) S + K_bar^T U (every warp, its 16 key channels) ----
        {
            const int m0 = 16 * warp;
            const float g0 = sGam[m0 + gq], g1 = sGam[m0 + gq + 8];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                Sf[nt][0] *= g0; Sf[nt][1] *= g0; Sf[nt][2] *= g1; Sf[nt][3] *= g1;
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                load_a_trans(sKb, LDK, m0, 16 * ks, lane, a);
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b[4];
                    load_b_kn(sK, LDK, 16 * np, 16 * ks, lane, b);
                    mma16816(Sf[2 * np], a, b[0], b[1]);
                    mma16816(Sf[2 * np + 1], a, b[2], b[3]);
                }
            }
        }
    }

    if (final_state) {
        float* sf = final_state + unit * (kDim * kDim);
        const int r0 = 16 * warp + gq;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            *reinterpret_cast<float2*>(sf + r0 * kDim + 8 * nt + 2 * tq) = make_float2(Sf[nt][0], Sf[nt][1]);
            *reinterpret_cast<float2*>(sf + (r0 + 8) * kDim + 8 * nt + 2 * tq) = make_float2(Sf[nt][2], Sf[nt][3]);
        }
    }
}

}  // namespace

cudaError_t launch_prefill(int dtype, int num_seqs, int heads, const void* q, const void* k,
                           const void* v, const void* g, const void* beta,
                           const float* init_state, const int32_t* cu_seqlens, void* out,
                           float* final_state, int* status, cudaStream_t stream,
                           uint64_t* launches) {
    if (num_seqs <= 0 || heads <= 0) return cudaSuccess;
    dim3 grid(num_seqs, heads);
    if (dtype == KDA_BF16) {
        using T = __nv_bfloat16;
        auto kern = kda_prefill_kernel<T>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, kSmemBytes, stream>>>(
            (const T*)q, (const T*)k, (const T*)v, (const T*)g, (const T*)beta, init_state,
            cu_seqlens, (T*)out, final_state, heads, status);
    } else {
        auto kern = kda_prefill_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, kSmemBytes, stream>>>(
            (const float*)q, (const float*)k, (const float*)v, (const float*)g,
            (const float*)beta, init_state, cu_seqlens, (float*)out, final_state, heads,
            status);
    }
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace kda
