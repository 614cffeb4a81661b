// kda_prefill_tc.cu — chunked KDA prefill on the sm_100-family tensor cores (tcgen05 + TMEM,
// TMA-fed), bf16 inputs, fp32 state.
//
// Method ("How Kimi K3 Engineered Its Way to the Frontier", section "FlashKDA steps the state
// once per 16 tokens"; the KDA recurrence from section "How KDA updates its state"): per
// 64-token chunk, aligned to the sequence start and zero-padded at the end, with
// G = within-chunk inclusive cumsum of g, G_C its last row and r = G_C / 2 per key channel:
//   Q_r = q e^{G-r}   K_p = k e^{G-r}   K_m = k e^{r-G}
//   A   = strict_lower(diag(beta) K_p K_m^T)   P = lower_incl(Q_r K_m^T)   T = (I + A)^{-1}
//   W   = T diag(beta) K_p                     U_bar = T diag(beta) V
//   X   = S^T diag(e^r)        (the state, transposed and column-scaled)
//   U^T = U_bar^T - X W^T      O^T = X Q_r^T + U^T P^T
//   S^T <- (X + U^T K_m) diag(e^r)
// (the last line is diag(e^{G_C}) S + K_bar^T U with K_bar = k e^{G_C-G} = K_m diag(e^r)).
//
// GB300 mapping.  One CTA per (sequence, head), 14 warps:
//   warp 0      TMA producer: q, k, g chunks into double-buffered slots; v single-buffered
//   warp 1      MMA issuer: one thread, event loop over six groups of tcgen05.mma
//   warps 2-9   prep: decay factors, A/P epilogue, 64x64 inverse, W epilogue (chunk c+1)
//   warps 10-13 serial epilogue: U^T to TMEM, O^T to HBM, state rescale (chunk c)
// so the chunk-parallel work of chunk c+1 overlaps the serial state pass of chunk c.  The
// state lives in TMEM (fp32, transposed so that value channels are TMEM lanes) for the whole
// sequence; its bf16 operand copy and U^T are also kept in TMEM and fed to the tensor core as
// the A operand, so no state byte goes through shared memory.  Every operand tile is used in
// the layout TMA or the producing warp writes naturally (K-major or MN-major 128B-swizzled).
//
// Precision: P, U and K_m enter the tensor core as two bf16 terms (hi + lo), which removes
// their rounding from the heavy tail of the output error; everything accumulates in fp32.
//
// Every wait is bounded; on expiry the CTA records KDA_ERR_TIMEOUT and drains.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;
using bf16 = __nv_bfloat16;

constexpr int kThreadsTC = 448;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpPrep0 = 2;   // 8 warps
constexpr int kWarpEpi0 = 10;   // 4 warps
constexpr int kPrepThreads = 256;
constexpr int kEpiThreads = 128;
constexpr int kBarPrep = 1;     // named barrier ids
constexpr int kBarEpi = 2;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s)
constexpr float kLog2eTC = 1.4426950408889634f;
constexpr float kMaxExponentTC = 80.f;
constexpr int LDA_T = 68;       // fp32 row stride of the 64 x 64 A / T matrix

// ---- shared memory map (bytes from a 1024-aligned base) ----
constexpr uint32_t OFF_KQ0 = 0;          // [K_p ; Q_r] slot 0: 128 rows x 128 cols (32 KB)
constexpr uint32_t OFF_KQ1 = 32768;      // slot 1
constexpr uint32_t OFF_KMH0 = 65536;     // K_m hi slot 0: 64 x 128 (16 KB)
constexpr uint32_t OFF_KMH1 = 81920;     // slot 1
constexpr uint32_t OFF_V = 98304;        // v: 64 x 128 (16 KB)
constexpr uint32_t OFF_P0 = 114688;      // P hi (8 KB) + P lo (8 KB), slot 0
constexpr uint32_t OFF_P1 = 131072;      // slot 1
constexpr uint32_t OFF_WN0 = 147456;     // g (as loaded), then -W^T: 128 x 64 (16 KB), slot 0
constexpr uint32_t OFF_WN1 = 163840;     // slot 1
constexpr uint32_t OFF_TB0 = 180224;     // T diag(beta): 64 x 64 (8 KB), slot 0
constexpr uint32_t OFF_TB1 = 188416;     // slot 1
constexpr uint32_t OFF_KML = 196608;     // K_m lo 64 x 128 (16 KB); after M1: A/T fp32 [64][68]
constexpr uint32_t OFF_Y = OFF_KML + 17408 + 1024;  // 3 x 16 x 16 fp32 block products
constexpr uint32_t OFF_BETA = OFF_Y + 3072;         // 64 fp32
constexpr uint32_t OFF_ER = OFF_BETA + 256;         // 4 x 128 fp32: e^{r} ring
constexpr uint32_t OFF_PART = OFF_ER + 2048;        // 2 x 128 fp32 partial sums
constexpr uint32_t OFF_BAR = OFF_PART + 1024;       // mbarriers
constexpr int NBAR = 24;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;   // tmem slot, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// barrier indices
enum {
    B_FULL0 = 0, B_FULL1, B_SLOTFREE0, B_SLOTFREE1, B_VFULL, B_VFREE,
    B_FACT0, B_FACT1, B_AP0, B_AP1, B_TB0, B_TB1, B_WDONE0, B_WDONE1, B_WN0, B_WN1,
    B_XDONE, B_UREADY, B_OSDONE, B_SREADY, B_DRAIN, B_COUNT
};
static_assert(B_COUNT <= NBAR, "barrier slots");

// TMEM columns (512 allocated)
constexpr uint32_t T_S = 0;      // X: fp32 state, lanes = value channel, cols = key channel
constexpr uint32_t T_O = 128;    // O^T (64 cols)
constexpr uint32_t T_U = 192;    // U^T (64 cols)
constexpr uint32_t T_P = 256;    // [A ; P] raw tiles, then W^T (64 cols)
constexpr uint32_t T_SA = 320;   // bf16 copy of X (A operand, 64 cols)
constexpr uint32_t T_UH = 384;   // bf16 U^T hi (A operand, 32 cols)
constexpr uint32_t T_UL = 416;   // bf16 U^T lo (32 cols)

struct TcParams {
    const bf16* beta;
    const float* init_state;
    const int32_t* cu_seqlens;
    bf16* out;
    float* final_state;
    int* status;
    int H;
};

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float bf2f(bf16 x) { return __bfloat162float(x); }

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimit) {
            *abort_flag = 1;
            report_status(status, kStatusTimeout);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreadsTC, 1)
kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g, const TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int n = blockIdx.x;
    const int h = blockIdx.y;
    const int H = p.H;
    const int64_t seq0 = p.cu_seqlens[n];
    const int L = p.cu_seqlens[n + 1] - (int)seq0;
    const int64_t unit = (int64_t)n * H + h;

    if (L <= 0) {  // empty sequence: the final state is the initial state
        if (p.final_state) {
            float* dst = p.final_state + unit * (kDim * kDim);
            const float* src = p.init_state ? p.init_state + unit * (kDim * kDim) : nullptr;
            for (int e = tid; e < kDim * kDim; e += blockDim.x) dst[e] = src ? src[e] : 0.f;
        }
        return;
    }
    const int nchunks = (L + kChunk - 1) / kChunk;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 8);
    float* beta_s = reinterpret_cast<float*>(sm + OFF_BETA);
    float* er = reinterpret_cast<float*>(sm + OFF_ER);
    float* part = reinterpret_cast<float*>(sm + OFF_PART);

    if (warp == kWarpTma) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_g);
            auto issue_kqg = [&](int c) {
                const int s = c & 1;
                unsigned char* kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
                unsigned char* wn = sm + (s ? OFF_WN1 : OFF_WN0);
                uint64_t* full = &bars[B_FULL0 + s];
                const int t0 = (int)(seq0 + (int64_t)kChunk * c);
                mbar_arrive_expect_tx(full, 49152);
                tma_load_3d(kq + 0, &tm_k, full, 0, h, t0);
                tma_load_3d(kq + 16384, &tm_k, full, 64, h, t0);
                tma_load_3d(kq + 8192, &tm_q, full, 0, h, t0);
                tma_load_3d(kq + 24576, &tm_q, full, 64, h, t0);
                tma_load_3d(wn + 0, &tm_g, full, 0, h, t0);
                tma_load_3d(wn + 8192, &tm_g, full, 64, h, t0);
            };
            auto issue_v = [&](int c) {
                const int t0 = (int)(seq0 + (int64_t)kChunk * c);
                mbar_arrive_expect_tx(&bars[B_VFULL], 16384);
                tma_load_3d(sm + OFF_V, &tm_v, &bars[B_VFULL], 0, h, t0);
                tma_load_3d(sm + OFF_V + 8192, &tm_v, &bars[B_VFULL], 64, h, t0);
            };
            issue_kqg(0);
            issue_v(0);
            if (nchunks > 1) issue_kqg(1);
            int next_kqg = 2, next_v = 1;
            long long last = clock64();
            while ((next_kqg < nchunks || next_v < nchunks) && !*abort_flag) {
                bool prog = false;
                if (next_v < nchunks && mbar_try_wait(&bars[B_VFREE], (next_v - 1) & 1)) {
                    issue_v(next_v++);
                    prog = true;
                }
                if (next_kqg < nchunks &&
                    mbar_try_wait(&bars[B_SLOTFREE0 + (next_kqg & 1)], ((next_kqg - 2) >> 1) & 1)) {
                    issue_kqg(next_kqg++);
                    prog = true;
                }
                if (prog) {
                    last = clock64();
                } else if (clock64() - last > kWaitLimit) {
                    *abort_flag = 1;
                    report_status(p.status, kStatusTimeout);
                }
            }
            if (*abort_flag) {
                // drain: let every issued copy land before the CTA can exit
                const int issued[2] = {(next_kqg + 1) / 2, next_kqg / 2};
                for (int s = 0; s < 2; ++s)
                    if (issued[s] > 0) mbar_wait(&bars[B_FULL0 + s], (issued[s] - 1) & 1, kWaitLimit);
                mbar_wait(&bars[B_VFULL], (next_v - 1) & 1, kWaitLimit);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t rS = tmem + T_S, rO = tmem + T_O, rU = tmem + T_U, rP = tmem + T_P;
            const uint32_t rSA = tmem + T_SA, rUH = tmem + T_UH, rUL = tmem + T_UL;
            const uint32_t a_kq[2] = {saddr(sm + OFF_KQ0), saddr(sm + OFF_KQ1)};
            const uint32_t a_kmh[2] = {saddr(sm + OFF_KMH0), saddr(sm + OFF_KMH1)};
            const uint32_t a_p[2] = {saddr(sm + OFF_P0), saddr(sm + OFF_P1)};
            const uint32_t a_wn[2] = {saddr(sm + OFF_WN0), saddr(sm + OFF_WN1)};
            const uint32_t a_tb[2] = {saddr(sm + OFF_TB0), saddr(sm + OFF_TB1)};
            const uint32_t a_kml = saddr(sm + OFF_KML), a_v = saddr(sm + OFF_V);
            const uint32_t id_kk64 = idesc_bf16(128, 64, false, false);
            const uint32_t id_mk64 = idesc_bf16(128, 64, true, false);
            const uint32_t id_km64 = idesc_bf16(128, 64, false, true);
            const uint32_t id_km128 = idesc_bf16(128, 128, false, true);
            int c1 = 0, c2 = 0, c3 = 0, c4 = 0, c56 = 0;
            long long last = clock64();
            while (c56 < nchunks && !*abort_flag) {
                bool prog = false;
                // M5 + M6: O^T += U^T P^T (3 split terms), X += U^T K_m (2 split terms)
                if (c56 < c4 && mbar_try_wait(&bars[B_UREADY], c56 & 1)) {
                    tc_fence_after();
                    const int s = c56 & 1;
                    for (int j = 0; j < 4; ++j)
                        mma_ts(rO, rUH + 8 * j, smem_desc(a_p[s] + 32 * j, 16, 1024), id_kk64, 1);
                    for (int j = 0; j < 4; ++j)
                        mma_ts(rO, rUL + 8 * j, smem_desc(a_p[s] + 32 * j, 16, 1024), id_kk64, 1);
                    for (int j = 0; j < 4; ++j)
                        mma_ts(rO, rUH + 8 * j, smem_desc(a_p[s] + 8192 + 32 * j, 16, 1024),
                               id_kk64, 1);
                    for (int j = 0; j < 4; ++j)
                        mma_ts(rS, rUH + 8 * j, smem_desc(a_kmh[s] + 2048 * j, 8192, 1024),
                               id_km128, 1);
                    for (int j = 0; j < 4; ++j)
                        mma_ts(rS, rUL + 8 * j, smem_desc(a_kmh[s] + 2048 * j, 8192, 1024),
                               id_km128, 1);
                    mma_commit(&bars[B_OSDONE]);
                    mma_commit(&bars[B_SLOTFREE0 + s]);
                    ++c56;
                    prog = true;
                }
                // M4: O^T = X Q_r^T, U^T += X (-W)^T
                if (c4 < c3 && c4 == c56 &&
                    mbar_try_wait(&bars[B_WN0 + (c4 & 1)], (c4 >> 1) & 1) &&
                    mbar_try_wait(&bars[B_SREADY], c4 & 1)) {
                    tc_fence_after();
                    const int s = c4 & 1;
                    for (int j = 0; j < 8; ++j)
                        mma_ts(rO, rSA + 8 * j,
                               smem_desc(a_kq[s] + 8192 + (j >> 2) * 16384 + (j & 3) * 32, 16, 1024),
                               id_kk64, j > 0);
                    for (int j = 0; j < 8; ++j)
                        mma_ts(rU, rSA + 8 * j, smem_desc(a_wn[s] + 2048 * j, 16384, 1024), id_km64,
                               1);
                    mma_commit(&bars[B_XDONE]);
                    ++c4;
                    prog = true;
                }
                // M3: U_bar^T = V^T (T diag(beta))^T
                if (c3 < c2 && c3 <= c56 && mbar_try_wait(&bars[B_VFULL], c3 & 1)) {
                    const int s = c3 & 1;
                    for (int j = 0; j < 4; ++j)
                        mma_ss(rU, smem_desc(a_v + 2048 * j, 8192, 1024),
                               smem_desc(a_tb[s] + 32 * j, 16, 1024), id_mk64, j > 0);
                    mma_commit(&bars[B_VFREE]);
                    ++c3;
                    prog = true;
                }
                // M2: W^T = K_p^T (T diag(beta))^T
                if (c2 < c1 && mbar_try_wait(&bars[B_TB0 + (c2 & 1)], (c2 >> 1) & 1)) {
                    tc_fence_after();
                    const int s = c2 & 1;
                    for (int j = 0; j < 4; ++j)
                        mma_ss(rP, smem_desc(a_kq[s] + 2048 * j, 16384, 1024),
                               smem_desc(a_tb[s] + 32 * j, 16, 1024), id_mk64, j > 0);
                    mma_commit(&bars[B_WDONE0 + s]);
                    ++c2;
                    prog = true;
                }
                // M1: [K_p ; Q_r] (K_m hi + K_m lo)^T
                if (c1 < nchunks && c1 <= c2 &&
                    mbar_try_wait(&bars[B_FACT0 + (c1 & 1)], (c1 >> 1) & 1)) {
                    tc_fence_after();
                    const int s = c1 & 1;
                    for (int j = 0; j < 8; ++j)
                        mma_ss(rP, smem_desc(a_kq[s] + (j >> 2) * 16384 + (j & 3) * 32, 16, 1024),
                               smem_desc(a_kmh[s] + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024),
                               id_kk64, j > 0);
                    for (int j = 0; j < 8; ++j)
                        mma_ss(rP, smem_desc(a_kq[s] + (j >> 2) * 16384 + (j & 3) * 32, 16, 1024),
                               smem_desc(a_kml + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024),
                               id_kk64, 1);
                    mma_commit(&bars[B_AP0 + s]);
                    ++c1;
                    prog = true;
                }
                if (prog) {
                    last = clock64();
                } else if (clock64() - last > kWaitLimit) {
                    *abort_flag = 1;
                    report_status(p.status, kStatusTimeout);
                }
            }
            // every issued MMA completes before TMEM can be released
            mma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, kWaitLimit);
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------------ prep (warps 2-9)
        const int tp = tid - kWarpPrep0 * 32;
        const int ch = tp & 127;
        const int half = tp >> 7;
        const int q4 = warp & 3;
        const int colhalf = (warp - kWarpPrep0) >> 2;
        const int row_abs = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        float* Am = reinterpret_cast<float*>(sm + OFF_KML);
        float* Y = reinterpret_cast<float*>(sm + OFF_Y);
        unsigned char* kml = sm + OFF_KML;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1;
            const int valid = min(kChunk, L - kChunk * c);
            const int64_t tok0 = seq0 + (int64_t)kChunk * c;
            unsigned char* kq = sm + (s ? OFF_KQ1 : OFF_KQ0);
            unsigned char* kmh = sm + (s ? OFF_KMH1 : OFF_KMH0);
            unsigned char* wn = sm + (s ? OFF_WN1 : OFF_WN0);
            unsigned char* pt = sm + (s ? OFF_P1 : OFF_P0);
            unsigned char* tb = sm + (s ? OFF_TB1 : OFF_TB0);
            float* ers = er + (c & 3) * kDim;
            if (!wait_bar(&bars[B_FULL0 + s], (c >> 1) & 1, abort_flag, p.status)) break;

            // ---- decay factors: two threads per key channel, 32 tokens each ----
            {
                float acc = 0.f;
#pragma unroll 8
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * half + i;
                    if (t < valid)
                        acc += bf2f(*reinterpret_cast<const bf16*>(wn + sw128_offset(t, ch, 64)));
                }
                part[half * kDim + ch] = acc;
                if (tp < kChunk)
                    beta_s[tp] = tp < valid ? bf2f(p.beta[(tok0 + tp) * H + h]) : 0.f;
            }
            named_bar(kBarPrep, kPrepThreads);
            {
                const float GC = part[ch] + part[kDim + ch];
                const float r = 0.5f * GC;
                float G = half ? part[ch] : 0.f;
                bool bad = false;
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * half + i;
                    const float gv =
                        t < valid ? bf2f(*reinterpret_cast<const bf16*>(wn + sw128_offset(t, ch, 64)))
                                  : 0.f;
                    G += gv;
                    const float d = G - r;
                    bad |= fabsf(d) > kMaxExponentTC;
                    const float e = exp2f(d * kLog2eTC);
                    const float ei = exp2f(-d * kLog2eTC);
                    bf16* pk = reinterpret_cast<bf16*>(kq + sw128_offset(t, ch, 128));
                    bf16* pq = reinterpret_cast<bf16*>(kq + sw128_offset(64 + t, ch, 128));
                    const float kv = bf2f(*pk), qv = bf2f(*pq);
                    *pk = __float2bfloat16_rn(kv * e);
                    *pq = __float2bfloat16_rn(qv * e);
                    const float km = kv * ei;
                    const bf16 kmh_v = __float2bfloat16_rn(km);
                    const uint32_t om = sw128_offset(t, ch, 64);
                    *reinterpret_cast<bf16*>(kmh + om) = kmh_v;
                    *reinterpret_cast<bf16*>(kml + om) = __float2bfloat16_rn(km - bf2f(kmh_v));
                }
                if (bad) report_status(p.status, kStatusDecayRange);
                if (half == 0) ers[ch] = exp2f(r * kLog2eTC);
            }
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_FACT0 + s]);

            // ---- A (rows 0-63) and P (rows 64-127) from TMEM ----
            if (!wait_bar(&bars[B_AP0 + s], (c >> 1) & 1, abort_flag, p.status)) break;
            tc_fence_after();
            {
                uint32_t v[32];
                tmem_ld32(tmem + T_P + 32 * colhalf + lane_off, v);
                if (row_abs < kChunk) {
                    const int t = row_abs;
                    const float bt = beta_s[t];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float4 o;
                        const int col = 32 * colhalf + 4 * j4;
                        o.x = col + 0 < t ? bt * __uint_as_float(v[4 * j4 + 0]) : 0.f;
                        o.y = col + 1 < t ? bt * __uint_as_float(v[4 * j4 + 1]) : 0.f;
                        o.z = col + 2 < t ? bt * __uint_as_float(v[4 * j4 + 2]) : 0.f;
                        o.w = col + 3 < t ? bt * __uint_as_float(v[4 * j4 + 3]) : 0.f;
                        *reinterpret_cast<float4*>(Am + t * LDA_T + col) = o;
                    }
                } else {
                    const int t = row_abs - kChunk;
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int col = 32 * colhalf + 8 * j8 + 2 * u;
                            const float x0 = col <= t ? __uint_as_float(v[8 * j8 + 2 * u]) : 0.f;
                            const float x1 = col + 1 <= t ? __uint_as_float(v[8 * j8 + 2 * u + 1]) : 0.f;
                            const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                            hi[u] = pack_bf16(bf2f(h0), bf2f(h1));
                            lo[u] = pack_bf16(x0 - bf2f(h0), x1 - bf2f(h1));
                        }
                        const uint32_t off = sw128_offset(t, 32 * colhalf + 8 * j8, 64);
                        *reinterpret_cast<uint4*>(pt + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(pt + 8192 + off) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
            tc_fence_before();
            named_bar(kBarPrep, kPrepThreads);

            // ---- T = (I + A)^{-1}: 16x16 diagonal blocks by forward substitution ----
            if (tp < 64) {
                const int b = tp >> 4, col = tp & 15;
                const float* Ab = Am + (16 * b) * LDA_T + 16 * b;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float sacc = (i == col) ? 1.f : 0.f;
#pragma unroll
                    for (int j = 0; j < i; ++j) sacc = fmaf(-Ab[i * LDA_T + j], x[j], sacc);
                    x[i] = sacc;
                }
                __syncwarp();
                float* Tb = Am + (16 * b) * LDA_T + 16 * b;
#pragma unroll
                for (int i = 0; i < 16; ++i) Tb[i * LDA_T + col] = x[i];
            }
            named_bar(kBarPrep, kPrepThreads);
            // ---- off-diagonal blocks: T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ ----
            for (int I = 1; I < 4; ++I) {
                for (int e = tp; e < I * 256; e += kPrepThreads) {
                    const int J = e >> 8, i = (e >> 4) & 15, j = e & 15;
                    float y = 0.f;
                    for (int K = J; K < I; ++K) {
                        const float* Arow = Am + (16 * I + i) * LDA_T + 16 * K;
                        const float* Tcol = Am + (16 * K) * LDA_T + 16 * J + j;
#pragma unroll
                        for (int x = 0; x < 16; ++x) y = fmaf(Arow[x], Tcol[x * LDA_T], y);
                    }
                    Y[e] = y;
                }
                named_bar(kBarPrep, kPrepThreads);
                for (int e = tp; e < I * 256; e += kPrepThreads) {
                    const int J = e >> 8, i = (e >> 4) & 15, j = e & 15;
                    const float* Trow = Am + (16 * I + i) * LDA_T + 16 * I;
                    const float* Ycol = Y + J * 256 + j;
                    float y = 0.f;
#pragma unroll
                    for (int x = 0; x < 16; ++x) y = fmaf(Trow[x], Ycol[x * 16], y);
                    Am[(16 * I + i) * LDA_T + 16 * J + j] = -y;
                }
                named_bar(kBarPrep, kPrepThreads);
            }
            // ---- T diag(beta) as the bf16 K-major operand ----
            for (int e = tp; e < kChunk * 8; e += kPrepThreads) {
                const int t = e >> 3, j8 = (e & 7) * 8;
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w[u] = pack_bf16(Am[t * LDA_T + j8 + 2 * u] * beta_s[j8 + 2 * u],
                                     Am[t * LDA_T + j8 + 2 * u + 1] * beta_s[j8 + 2 * u + 1]);
                *reinterpret_cast<uint4*>(tb + sw128_offset(t, j8, 64)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_TB0 + s]);

            // ---- -W^T into the [c][t] operand tile ----
            if (!wait_bar(&bars[B_WDONE0 + s], (c >> 1) & 1, abort_flag, p.status)) break;
            tc_fence_after();
            {
                uint32_t v[32];
                tmem_ld32(tmem + T_P + 32 * colhalf + lane_off, v);
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        w[u] = pack_bf16(-__uint_as_float(v[8 * j8 + 2 * u]),
                                         -__uint_as_float(v[8 * j8 + 2 * u + 1]));
                    *reinterpret_cast<uint4*>(wn + sw128_offset(row_abs, 32 * colhalf + 8 * j8, 128)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            tc_fence_before();
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_WN0 + s]);
        }
    } else {
        // ------------------------------------------------------------ serial epilogue
        const int te = tid - kWarpEpi0 * 32;
        const int q4 = warp & 3;
        const int vch = 32 * q4 + lane;  // value channel = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        bool ok = wait_bar(&bars[B_FACT0], 0, abort_flag, p.status);
        if (ok) {  // X_0 = S0^T diag(e^{r_0})
            const float* e0 = er;
            const float* s0 = p.init_state ? p.init_state + unit * (kDim * kDim) : nullptr;
            for (int cc = 0; cc < kDim; cc += 32) {
                uint32_t x[32], xb[16];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sv = s0 ? s0[(cc + j) * kDim + vch] : 0.f;
                    x[j] = __float_as_uint(sv * e0[cc + j]);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    xb[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
                tmem_st32(tmem + T_S + cc + lane_off, x);
                tmem_st16(tmem + T_SA + cc / 2 + lane_off, xb);
            }
            tmem_st_wait();
            tc_fence_before();
            named_bar(kBarEpi, kEpiThreads);
            if (te == 0) mbar_arrive(&bars[B_SREADY]);
        }
        for (int c = 0; ok && c < nchunks; ++c) {
            const int valid = min(kChunk, L - kChunk * c);
            const int64_t tok0 = seq0 + (int64_t)kChunk * c;
            // ---- E1: U^T -> bf16 hi/lo A operands ----
            if (!(ok = wait_bar(&bars[B_XDONE], c & 1, abort_flag, p.status))) break;
            tc_fence_after();
            {
                uint32_t u[32], hi[32], lo[32];
#pragma unroll
                for (int g2 = 0; g2 < 2; ++g2) {
                    tmem_ld32(tmem + T_U + 32 * g2 + lane_off, u);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float x0 = __uint_as_float(u[2 * j]), x1 = __uint_as_float(u[2 * j + 1]);
                        const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                        hi[16 * g2 + j] = pack_bf16(bf2f(h0), bf2f(h1));
                        lo[16 * g2 + j] = pack_bf16(x0 - bf2f(h0), x1 - bf2f(h1));
                    }
                }
                tmem_st32(tmem + T_UH + lane_off, hi);
                tmem_st32(tmem + T_UL + lane_off, lo);
                tmem_st_wait();
            }
            tc_fence_before();
            named_bar(kBarEpi, kEpiThreads);
            if (te == 0) mbar_arrive(&bars[B_UREADY]);

            // ---- E2: O to HBM, state rescale ----
            if (!(ok = wait_bar(&bars[B_OSDONE], c & 1, abort_flag, p.status))) break;
            tc_fence_after();
            {
                uint32_t o[32];
#pragma unroll
                for (int g2 = 0; g2 < 2; ++g2) {
                    tmem_ld32(tmem + T_O + 32 * g2 + lane_off, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = 32 * g2 + j;
                        if (t < valid)
                            p.out[((tok0 + t) * H + h) * kDim + vch] =
                                __float2bfloat16_rn(__uint_as_float(o[j]));
                    }
                }
            }
            const float* ec = er + (c & 3) * kDim;
            if (c + 1 < nchunks) {
                if (!(ok = wait_bar(&bars[B_FACT0 + ((c + 1) & 1)], ((c + 1) >> 1) & 1, abort_flag,
                                    p.status)))
                    break;
                const float* en = er + ((c + 1) & 3) * kDim;
                for (int cc = 0; cc < kDim; cc += 32) {
                    uint32_t x[32], xb[16];
                    tmem_ld32(tmem + T_S + cc + lane_off, x);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        x[j] = __float_as_uint(__uint_as_float(x[j]) * (ec[cc + j] * en[cc + j]));
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        xb[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
                    tmem_st32(tmem + T_S + cc + lane_off, x);
                    tmem_st16(tmem + T_SA + cc / 2 + lane_off, xb);
                }
                tmem_st_wait();
                tc_fence_before();
                named_bar(kBarEpi, kEpiThreads);
                if (te == 0) mbar_arrive(&bars[B_SREADY]);
            } else if (p.final_state) {
                float* fs = p.final_state + unit * (kDim * kDim);
                for (int cc = 0; cc < kDim; cc += 32) {
                    uint32_t x[32];
                    tmem_ld32(tmem + T_S + cc + lane_off, x);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        fs[(cc + j) * kDim + vch] = __uint_as_float(x[j]) * ec[cc + j];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpTma) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over [T_tot, H, 128] bf16 (innermost first), box = 64 channels x 1 head x 64 tokens.
bool make_map(CUtensorMap* map, const void* base, int64_t T, int H) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)H * kDim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_tc(int num_seqs, int heads, int64_t total_tokens, const void* q,
                              const void* k, const void* v, const void* g, const void* beta,
                              const float* init_state, const int32_t* cu_seqlens, void* out,
                              float* final_state, int* status, cudaStream_t stream,
                              uint64_t* launches) {
    if (num_seqs <= 0 || heads <= 0) return cudaSuccess;
    CUtensorMap mq, mk, mv, mg;
    const int64_t T = total_tokens > 0 ? total_tokens : 1;
    if (!make_map(&mq, q, T, heads) || !make_map(&mk, k, T, heads) ||
        !make_map(&mv, v, T, heads) || !make_map(&mg, g, T, heads))
        return cudaErrorInvalidValue;
    TcParams prm;
    prm.beta = static_cast<const bf16*>(beta);
    prm.init_state = init_state;
    prm.cu_seqlens = cu_seqlens;
    prm.out = static_cast<bf16*>(out);
    prm.final_state = final_state;
    prm.status = status;
    prm.H = heads;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    dim3 grid(num_seqs, heads);
    kda_prefill_tc_kernel<<<grid, kThreadsTC, SMEM_ALLOC, stream>>>(mq, mk, mv, mg, prm);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace kda
