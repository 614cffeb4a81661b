// kda_prefill_tc.cu — chunked KDA prefill on the sm_100-family tensor cores (tcgen05 + TMEM,
// TMA-fed), bf16 inputs, fp32 state.
//
// Method ("How Kimi K3 Engineered Its Way to the Frontier", section "FlashKDA steps the state
// once per 16 tokens"; the KDA recurrence from section "How KDA updates its state"): per
// chunk of at most 64 tokens, zero-padded at the end, with G = within-chunk inclusive cumsum of
// g, G_C its last row and r = G_C / 2 per key channel:
//   Q_r = q e^{G-r}   K_p = k e^{G-r}   K_m = k e^{r-G}
//   A   = strict_lower(diag(beta) K_p K_m^T)   P = lower_incl(Q_r K_m^T)   T = (I + A)^{-1}
//   W   = T diag(beta) K_p                     U_bar = T diag(beta) V
//   X   = S^T diag(e^r)        (the state, transposed and column-scaled)
//   U^T = U_bar^T - X W^T      O^T = X Q_r^T + U^T P^T
//   S^T <- (X + U^T K_m) diag(e^r)
// (the last line is diag(e^{G_C}) S + K_bar^T U with K_bar = k e^{G_C-G} = K_m diag(e^r)).
//
// Decay windows.  Every factor above is an exponential of |G - r| <= |G_C| / 2, and the state
// scale between chunks is e^{r_{c-1} + r_c}; all stay normal fp32 (and bf16) numbers when
// |G_C| <= 80 in every channel.  The bounded gate allows up to 5 per token, 320 over 64 tokens,
// so a chunk is a window of the sequence: it starts where the previous one ended, never
// crosses a multiple of 64 tokens from the sequence start, and is the longest run of whole
// four-token groups (or the rest of the 64-token block) whose decay stays within 80 in every
// channel.  With ordinary gates every window is a whole 64-token block; a block that decays
// faster runs as two to sixteen windows, each through the same pipeline (its tiles are loaded
// from the window's first token and the rows past its end are masked as padding).  A
// four-token group that alone decays by more than 80 (log_alpha below -20) is reported as
// KDA_ERR_DECAY_RANGE, as is a positive log_alpha.
//
// GB300 mapping.  One CTA per (sequence, head), 14 warps:
//   warp 0      prep MMA issuer (one thread): the chunk-local products of chunk c+1, the TMA
//               loads of v and of g one chunk ahead; it also issues the first q, k, g, v loads
//   warp 1      serial MMA issuer (one thread): the state products of chunk c
//   warps 2-9   prep: exponential factors, A/P epilogue, 64x64 inverse, W epilogue (chunk c+1)
//   warps 10-13 serial epilogue: U^T to TMEM, the cumulative decay of chunk c+2, state rescale,
//               O^T to HBM (chunk c), and the k, q refill of chunk c+2
// so the chunk-parallel work of chunk c+1 overlaps the serial state pass of chunk c.  The
// state lives in TMEM (fp32, transposed so that value channels are TMEM lanes) for the whole
// sequence; its bf16 operand copy and U^T are also kept in TMEM and fed to the tensor core as
// the A operand, so no state byte goes through shared memory.  Every operand tile is used in
// the layout TMA or the producing warp writes naturally (K-major or MN-major 128B-swizzled).
//
// Precision: P and U enter the tensor core as two bf16 terms (hi + lo), which removes their
// rounding from the heavy tail of the output error; everything accumulates in fp32.  Two terms
// that fast decay makes dominant get more: in a chunk whose decay exceeds kHeavyDecay in some
// channel, P's diagonal q_t . k_t (its decay factor is exactly 1) is formed in fp32 from the
// raw tiles rather than from the bf16-rounded factor tiles; and the state update of a work
// item's last chunk (the state it returns) adds K_m's bf16 rounding residue as a third term.
//
// Every wait is bounded; on expiry the CTA records KDA_ERR_TIMEOUT and drains.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"
#include "kda_prologue.cuh"
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
constexpr float kWindowDecay = 80.f;  // largest |G_C| of a window (so |G - r| <= 40)
constexpr float kHeavyDecay = 48.f;   // chunks decaying faster in some channel form P's diagonal
                                      // from the raw q, k (it then dominates the output)
constexpr int kWinRing = 8;     // window records kept: the oldest reader is two chunks behind
constexpr int LDA_T = 68;       // fp32 row stride of the 64 x 64 A / T matrix

// ---- shared memory map (bytes from a 1024-aligned base) ----
// Slot tile [k -> K_p -> -W ; q -> Q_r]: 128 rows x 128 cols, two column regions of 16 KB.  It
// is the A operand of the intra-chunk product ([K_p ; Q_r]) and later the B operand of the state
// product ([-W ; Q_r], -W written over K_p once M2 has read it); k and q of chunk c + 2 wait for
// M4 of chunk c.  g has one buffer of its own: only the decay scan and the factor pass read it,
// so g of chunk c + 1 is loaded as soon as the factor pass of chunk c is done.  K_m has three
// slots, so the factor pass of chunk c waits for M6 of chunk c - 3 rather than c - 2.
constexpr int KQW_ROWS = 128;
constexpr uint32_t KQW_REGION = KQW_ROWS * 128;   // 16384
constexpr uint32_t OFF_KQW0 = 0;         // slot 0 (32 KB)
constexpr uint32_t OFF_KQW1 = 32768;     // slot 1
constexpr uint32_t OFF_G = 65536;        // g: 64 x 128 (16 KB), two column regions of 8 KB
constexpr uint32_t OFF_KMH0 = 81920;     // K_m slot 0: 64 x 128 (16 KB)
constexpr uint32_t OFF_KMH1 = 98304;     // slot 1
constexpr uint32_t OFF_KMH2 = 114688;    // slot 2
constexpr uint32_t OFF_V = 131072;       // v: 64 x 128 (16 KB)
constexpr uint32_t OFF_P0 = 147456;      // P hi (8 KB) + P lo (8 KB), slot 0
constexpr uint32_t OFF_P1 = 163840;      // slot 1
constexpr uint32_t OFF_TB0 = 180224;     // T diag(beta): 64 x 64 (8 KB), slot 0
constexpr uint32_t OFF_TB1 = 188416;     // slot 1
constexpr uint32_t OFF_KML = 196608;     // A / T fp32 [64][68] of the 64 x 64 inverse
constexpr uint32_t OFF_PART = OFF_KML + 17408;      // 16 x 128 fp32 token-group prefixes
constexpr uint32_t OFF_GC = OFF_PART + 8192;        // 128 fp32: chunk log-decay G_C
constexpr uint32_t OFF_BETA = OFF_GC + 512;         // 2 x 64 fp32 ring
constexpr uint32_t OFF_ER = OFF_BETA + 512;         // 4 x 128 fp32: e^{r} ring
constexpr uint32_t OFF_SC = OFF_ER + 2048;          // 4 x 128 fp32: e^{r_{c-1} + r_c} ring
constexpr uint32_t OFF_BAR = OFF_SC + 2048;         // mbarriers
constexpr int NBAR = 36;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;   // tmem slot, abort flag, copies issued
constexpr uint32_t OFF_WIN = OFF_MISC + 48;         // kWinRing x {first token, length, fast, 0}
constexpr uint32_t OFF_WMIN = OFF_WIN + kWinRing * 16;  // 4 ints: per-warp window group counts
constexpr uint32_t OFF_QK = OFF_WMIN + 16;         // 4 x 64 fp32: q_t . k_t by chunk (P's diagonal)
constexpr uint32_t OFF_HEAVY = OFF_QK + 1024;       // 4 ints: per-warp flags of the rare path
constexpr uint32_t SMEM_USED = OFF_HEAVY + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// barrier indices
enum {
    B_FULL0 = 0, B_FULL1, B_VFREE0, B_VFREE1, B_VFULL, B_SPARE,
    B_FACT0, B_FACT1, B_AP0, B_AP1, B_TB0, B_TB1, B_WDONE0, B_WDONE1, B_WN0, B_WN1,
    B_XDONE, B_UREADY, B_OSDONE, B_SREADY, B_DRAIN, B_UFREE0, B_UFREE1, B_KMFREE0, B_KMFREE1, B_KMFREE2,
    B_SDONE, B_PFREE0, B_PFREE1, B_SCAN0, B_SCAN1, B_GFULL, B_M6ISS,
    B_VPRO,  // prologue variant: v of the chunk has been through Swish
    B_KQPRO0, B_KQPRO1,  // prologue variant: k, q of the slot are transformed (one per prep warp)
    B_COUNT
};
static_assert(B_COUNT <= NBAR, "barrier slots");

// TMEM columns (512 allocated)
constexpr uint32_t T_S = 0;      // X: fp32 state, lanes = value channel, cols = key channel
constexpr uint32_t T_X0 = 128;   // even chunks: [U^T (64) | O^T (64)]; U^T becomes bf16 hi|lo;
                                 // the O^T columns first hold W^T of the chunk
constexpr uint32_t T_P = 256;    // [A ; P] raw tiles (64 cols)
constexpr uint32_t T_SA = 320;   // bf16 copy of X (A operand, 64 cols)
constexpr uint32_t T_X1 = 384;   // odd chunks

struct TcParams {
    const bf16* beta;
    const float* init_state;
    const int32_t* cu_seqlens;
    bf16* out;
    float* final_state;
    int* status;
    float* ws_tilde;   // segment states from zero        [slots][H][128][128]
    float* ws_trans;   // segment transitions             [slots][H][128][128]
    float* ws_in;      // composed incoming states        [slots][H][128][128]
    float* ckpt;       // state checkpoints [count][H][128][128], or null
    int ckpt_chunks;   // chunks between checkpoints
    int H;
    int pass;          // 0: whole sequences + pass A of split ones; 1: pass B of split ones
    // input prologue (the kPro variant): q, k, v, g, beta are raw projections
    const float* pro_A_log;    // [H]
    const float* pro_dt_bias;  // [H][128] or null
    float pro_lb;              // lower bound of log alpha
    float pro_q_scale;
};

// What one CTA does (chosen from the sequence length and blockIdx.z).
enum { ITEM_WHOLE = 0, ITEM_TILDE = 1, ITEM_TRANS = 2, ITEM_SEGMENT = 3 };

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also returns whether `pred` holds in any participating thread.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}


__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}

// ---- 16 x 16 fp32 block products on the tensor cores (tf32 inputs, fp32 accumulate) ----
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc += (xs * X + n2 - n3) Yb for 16 x 16 blocks; n2 / n3 (leading dim LDA_T) may be null.
// Four 8 x 4 fp32 tiles (as 8 x 8 b16 matrices) in one instruction: lane l gives the address
// of row l & 7 of tile l >> 3, and register i of lane l receives tile i's element
// (l / 4, l % 4).  Rows must start on 16-byte boundaries.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const float* row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr(row))
                 : "memory");
}
// acc += (xs X + n2 - n3) Yb for 16 x 16 blocks (n2, n3 optional, stride LDA_T).  The A fragments
// (rows g, g + 8; columns k0 + t, k0 + t + 4) come from ldmatrix: tiles (rows 0-7 | 8-15) x
// (columns k0..k0+3 | k0+4..k0+7).
__device__ __forceinline__ void block_mma(float (&acc)[2][4], const float* X, int ldx, float xs,
                                          const float* n2, const float* n3, const float* Yb,
                                          int ldy, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int mrow = (lane & 7) + ((lane & 8) ? 8 : 0), mcol = (lane & 16) ? 4 : 0;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int k0 = 8 * ks;
        uint32_t a[4];
        ldsm_x4(a, X + mrow * ldx + k0 + mcol);
        uint32_t a2[4] = {0u, 0u, 0u, 0u}, a3[4] = {0u, 0u, 0u, 0u};
        if (n2) ldsm_x4(a2, n2 + mrow * LDA_T + k0 + mcol);
        if (n3) ldsm_x4(a3, n3 + mrow * LDA_T + k0 + mcol);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float x = xs * __uint_as_float(a[i]);
            if (n2) x += __uint_as_float(a2[i]);
            if (n3) x -= __uint_as_float(a3[i]);
            a[i] = to_tf32(x);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int n0 = 8 * nt;
            mma_tf32(acc[nt], a, to_tf32(Yb[(k0 + t) * ldy + n0 + g]),
                     to_tf32(Yb[(k0 + t + 4) * ldy + n0 + g]));
        }
    }
}
__device__ __forceinline__ void block_product(float (&acc)[2][4], const float* X, int ldx, float xs,
                                              const float* n2, const float* n3, const float* Yb,
                                              int ldy, int lane) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    block_mma(acc, X, ldx, xs, n2, n3, Yb, ldy, lane);
}
__device__ __forceinline__ void store_block(float* D, int ld, const float (&acc)[2][4], int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(D + g * ld + 8 * nt + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(D + (g + 8) * ld + 8 * nt + 2 * t) =
            make_float2(acc[nt][2], acc[nt][3]);
    }
}
// Block (I, J) of T diag(beta) as bf16 into the 64 x 64 128B-swizzled operand tile.
__device__ __forceinline__ void store_block_tb(unsigned char* tb, int I, int J,
                                               const float (&acc)[2][4], const float* beta_s,
                                               int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int col = 16 * J + 8 * nt + 2 * t;
        const float b0 = beta_s[col], b1 = beta_s[col + 1];
        *reinterpret_cast<uint32_t*>(tb + sw128_offset(16 * I + g, col, 64)) =
            pack_bf16(acc[nt][0] * b0, acc[nt][1] * b1);
        *reinterpret_cast<uint32_t*>(tb + sw128_offset(16 * I + g + 8, col, 64)) =
            pack_bf16(acc[nt][2] * b0, acc[nt][3] * b1);
    }
}
// block pairs (I, J), I > J, of the 4 x 4 block-lower 64 x 64 matrix, one per prep warp
__device__ __forceinline__ int pair_i(int w) { return w < 1 ? 1 : (w < 3 ? 2 : 3); }
__device__ __forceinline__ int pair_j(int w) { const int I = pair_i(w); return w - I * (I - 1) / 2; }

__device__ __noinline__ bool wait_bar_poll(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag, int* status) {
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
// Wait for a barrier phase; the polling loop is out of line to keep the kernel's code small.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
    return mbar_try_wait(bar, parity) || wait_bar_poll(bar, parity, abort_flag, status);
}

// The issuer threads' wait: a first non-blocking probe, then the same try_wait loop as the
// other warps (measured: no slower than shorter suspend hints or a test_wait spin).
__device__ __noinline__ bool spin_bar_poll(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag, int* status) {
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
__device__ __forceinline__ bool spin_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
    return mbar_test(bar, parity) || spin_bar_poll(bar, parity, abort_flag, status);
}

// The state after a chunk for one warp's 32 value channels: S[k][v] = X[v][k] e^{r_k} with X
// read from TMEM at taddr (the warp's lanes, key channels as columns); dst is [128][128] fp32,
// row = key channel.
__device__ __forceinline__ void store_state(float* dst, uint32_t taddr, const float* ec, int vch) {
#pragma unroll 1
    for (int cc = 0; cc < kDim; cc += 32) {
        uint32_t x[32];
        tmem_ld32(taddr + cc, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(cc + j) * kDim + vch] = __uint_as_float(x[j]) * ec[cc + j];
    }
}

// Shorten chunk cs's window when some channel's decay over the vmax tokens the scan covered
// exceeds the bound: nok is this channel's count of leading four-token groups within it, and
// the smallest count over the channels, nmin, sets the window's length 4 nmin.  Tokens past the
// window count as padding (g = 0), so the prefixes of later groups, G_C, e^{r} and the state
// scale become those of the window.  Each thread rewrites its own channel's entries.  Inlined
// into the (out-of-line) scan: a call there would make every scan save registers.
__device__ __forceinline__ int shorten_window(unsigned char* sm, int cs, int te, int nok, int vmax,
                                           int* status) {
    float* part = reinterpret_cast<float*>(sm + OFF_PART);
    float* gc_s = reinterpret_cast<float*>(sm + OFF_GC);
    float* er = reinterpret_cast<float*>(sm + OFF_ER);
    float* sc = reinterpret_cast<float*>(sm + OFF_SC);
    int* wmin = reinterpret_cast<int*>(sm + OFF_WMIN);
    const int wm = (int)__reduce_min_sync(0xffffffffu, (unsigned)nok);
    if ((te & 31) == 0) wmin[te >> 5] = wm;
    named_bar(kBarEpi, kEpiThreads);
    const int4 m4 = *reinterpret_cast<const int4*>(wmin);
    int nmin = min(min(m4.x, m4.y), min(m4.z, m4.w));
    if (nmin == 0) {  // one four-token group alone decays beyond the range: log_alpha < -20
        if (te == 0) report_status(status, kStatusDecayRange);
        nmin = 1;
    }
    const int len = min(vmax, 4 * nmin);
    if (len < vmax) {
        const float G = part[nmin * kDim + te];  // decay after the window's 4 nmin tokens
#pragma unroll 1
        for (int gi = nmin + 1; gi < 16; ++gi) part[gi * kDim + te] = G;
        gc_s[te] = G;
        const float e = ex2_approx((0.5f * kLog2eTC) * G);
        er[(cs & 3) * kDim + te] = e;
        sc[(cs & 3) * kDim + te] = cs > 0 ? er[((cs + 3) & 3) * kDim + te] * e : e;
    }
    named_bar(kBarEpi, kEpiThreads);
    return len;
}

// The extra terms of chunk cs, for the chunks that need them (inlined into the scan, which the
// factor pass of the chunk waits for; thread te of the epilogue group):
//   heavy: q_t . k_t in fp32 from the chunk's bf16 k and q tiles (thread t < 64), for P's
//          diagonal: under fast decay that term dominates o_t;
//   last:  the work item's last chunk: K_m's bf16 rounding residue k e^{r-G} - K_m (column te),
//          with the factor pass's own arithmetic for K_m, into the K_m slot after this chunk's
//          (free once M6 of chunk cs - 2 has read it), for a third term of the final state update.
// The k, q tiles are read before the factor pass replaces them (it waits for the scan).
template <bool kPro>
__device__ __forceinline__ bool scan_extra(unsigned char* sm, int cs, int te, int len, bool heavy,
                                           bool last, volatile int* abort_flag, int* status) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    const int s2 = cs & 1;
    // k and q of the chunk have landed (the prologue variant: and are transformed)
    if (!wait_bar(&bars[(kPro ? B_KQPRO0 : B_FULL0) + s2], (cs >> 1) & 1, abort_flag, status))
        return false;
    const unsigned char* kq = sm + (s2 ? OFF_KQW1 : OFF_KQW0);
    if (heavy && te < kChunk) {
        float d = 0.f;
#pragma unroll 4
        for (int c8 = 0; c8 < kDim; c8 += 8) {
            const uint32_t o = sw128_offset(te, c8, KQW_ROWS);
            float kv[8], qv[8];
            unpack8(*reinterpret_cast<const uint4*>(kq + o), kv);
            unpack8(*reinterpret_cast<const uint4*>(kq + o + 64 * 128), qv);
#pragma unroll
            for (int j = 0; j < 8; ++j) d = fmaf(qv[j], kv[j], d);
        }
        reinterpret_cast<float*>(sm + OFF_QK)[(cs & 3) * kChunk + te] = d;
    }
    if (last) {
        const int sl = (cs + 1) % 3;
        if (cs >= 2 && !wait_bar(&bars[B_KMFREE0 + sl], ((cs - 2) / 3) & 1, abort_flag, status))
            return false;
        unsigned char* dst = sm + (sl == 0 ? OFF_KMH0 : sl == 1 ? OFF_KMH1 : OFF_KMH2);
        const float* part = reinterpret_cast<const float*>(sm + OFF_PART);
        const float r = (0.5f * kLog2eTC) * reinterpret_cast<const float*>(sm + OFF_GC)[te];
#pragma unroll 1
        for (int tg = 0; tg < 16; ++tg) {
            float G = fmaf(part[tg * kDim + te], kLog2eTC, -r);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * tg + i;
                const float gv = t < len ? __bfloat162float(*reinterpret_cast<const bf16*>(
                                               sm + OFF_G + sw128_offset(t, te, 64)))
                                         : 0.f;
                G = fmaf(gv, kLog2eTC, G);
                const float km = __bfloat162float(*reinterpret_cast<const bf16*>(
                                     kq + sw128_offset(t, te, KQW_ROWS))) *
                                 ex2_approx(-G);
                *reinterpret_cast<bf16*>(dst + sw128_offset(t, te, 64)) =
                    __float2bfloat16_rn(km - round_bf16(km));
            }
        }
        fence_async_shared();  // read by the tensor core
    }
    named_bar(kBarEpi, kEpiThreads);
    return true;
}

// Cumulative decay of chunk cs for the epilogue warp group, thread te = key channel: the
// chunk's window (first token and length), the exclusive prefixes of g at its 16 four-token
// groups (into the prefix array), G_C, e^{r} with r = G_C / 2, and the state scale
// e^{r_{cs-1} + r_cs}.  Group sums first, then the prefix over the groups.  The window starts
// where chunk cs - 1's ended and first covers the rest of its 64-token block (the g tile was
// loaded from its first token); each channel counts the leading groups whose prefix stays
// within kWindowDecay, and the smallest count over the channels sets the window's length.
// One call site, out of line: inlined, it raises the epilogue loop's spills.
// kPro: g is the raw gate input; each value goes through the bounded gate (rounded to bf16, as
// an unfused prologue would store it) and is written back for the factor pass.
// Returns -1 when a wait gave up, 0 when the chunk is released (the common case), or 1 when
// the chunk needs the rare path (scan_rare: a shorter window, or the extra terms).
template <bool kPro>
__device__ __forceinline__ int decay_scan_body(unsigned char* sm, int cs, int L, int te,
                                               volatile int* abort_flag, int* status, float dt,
                                               float a, float lb) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    float* part = reinterpret_cast<float*>(sm + OFF_PART);
    float* gc_s = reinterpret_cast<float*>(sm + OFF_GC);
    float* er = reinterpret_cast<float*>(sm + OFF_ER);
    float* sc = reinterpret_cast<float*>(sm + OFF_SC);
    int4* win = reinterpret_cast<int4*>(sm + OFF_WIN);
    const int s2 = cs & 1;
    const int t0 = cs == 0 ? 0 : win[(cs - 1) & (kWinRing - 1)].x + win[(cs - 1) & (kWinRing - 1)].y;
    const int vmax = min(L - t0, kChunk - (t0 & (kChunk - 1)));
    if (!wait_bar(&bars[B_GFULL], cs & 1, abort_flag, status)) return -1;
    // g of token t is row t of its column region
    const unsigned char* gcol = sm + OFF_G + (te >> 6) * 8192 + ((te & 7) << 1);
    const int chunk16 = (te & 63) >> 3;
    float run = 0.f, gmax = 0.f;
#pragma unroll 1
    for (int t16 = 0; t16 < kChunk; t16 += 16) {
        // sixteen tokens' loads in flight at once; rows past the window hold other tokens (or
        // zeros) and are masked after the load
        float gv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            gv[i] = __bfloat162float(*reinterpret_cast<const bf16*>(
                gcol + (t16 + i) * 128 + ((chunk16 ^ (i & 7)) << 4)));
        if constexpr (kPro) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float2 gg = pro_gate2(make_float2(gv[i], gv[i + 1]), dt, a, lb);
                gv[i] = gg.x;
                gv[i + 1] = gg.y;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<bf16*>(const_cast<unsigned char*>(gcol) + (t16 + i) * 128 +
                                         ((chunk16 ^ (i & 7)) << 4)) = __float2bfloat16_rn(gv[i]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float gs = 0.f;
#pragma unroll
            for (int i = 4 * q; i < 4 * q + 4; ++i) {
                const float x = t16 + i < vmax ? gv[i] : 0.f;  // g is zero past the window
                gs += x;
                gmax = fmaxf(gmax, x);
            }
            part[((t16 >> 2) + q) * kDim + te] = run;
            run += gs;
        }
    }
    if (gmax > 0.f) report_status(status, kStatusDecayRange);
    const bool heavy = fabsf(run) > kHeavyDecay;  // this channel decays fast
    gc_s[te] = run;
    const float e = ex2_approx((0.5f * kLog2eTC) * run);
    er[(cs & 3) * kDim + te] = e;
    sc[(cs & 3) * kDim + te] = cs > 0 ? er[((cs + 3) & 3) * kDim + te] * e : e;
    if constexpr (kPro) fence_async_shared();  // the gated g is overwritten by the next TMA load
    // the barrier tells every thread whether some channel needs the rare path: fast decay
    // (which includes every window that must be shortened, as kWindowDecay > kHeavyDecay); the
    // item's last chunk takes it too
    if (named_bar_or(kBarEpi, kEpiThreads, heavy) || t0 + vmax >= L) return 1;
    if (te == 0) {
        win[cs & (kWinRing - 1)] = make_int4(t0, vmax, 0, 0);
        mbar_arrive(&bars[B_SCAN0 + s2]);
    }
    return 0;
}

// The rare path of chunk cs's scan, out of line so that the common scan stays small: shorten
// the window if some channel needs it, add the extra terms for a fast-decaying chunk or the
// item's last chunk, then release the chunk.
template <bool kPro>
__device__ __forceinline__ bool scan_rare_body(unsigned char* sm, int cs, int L, int te,
                                               volatile int* abort_flag, int* status) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    int4* win = reinterpret_cast<int4*>(sm + OFF_WIN);
    int* flags = reinterpret_cast<int*>(sm + OFF_HEAVY);
    const float* part = reinterpret_cast<const float*>(sm + OFF_PART);
    const float gc = reinterpret_cast<const float*>(sm + OFF_GC)[te];
    const int t0 = cs == 0 ? 0 : win[(cs - 1) & (kWinRing - 1)].x + win[(cs - 1) & (kWinRing - 1)].y;
    const int vmax = min(L - t0, kChunk - (t0 & (kChunk - 1)));
    // this channel's leading four-token groups whose decay stays within the window bound (the
    // prefix after group i is the exclusive prefix of group i + 1); |G| only grows, as g <= 0
    int nok = 0;
#pragma unroll 1
    for (int gi = 1; gi <= 16; ++gi)
        nok += fabsf(gi < 16 ? part[gi * kDim + te] : gc) <= kWindowDecay ? 1 : 0;
    // per warp: bit 0 some channel decays fast, bit 1 the window must be shorter than vmax
    const unsigned heavy = __any_sync(0xffffffffu, fabsf(gc) > kHeavyDecay);
    const unsigned shrt = __any_sync(0xffffffffu, 4 * nok < vmax);
    if ((te & 31) == 0) flags[te >> 5] = (heavy ? 1 : 0) | (shrt ? 2 : 0);
    named_bar(kBarEpi, kEpiThreads);
    const int4 f = *reinterpret_cast<const int4*>(flags);
    const int fo = f.x | f.y | f.z | f.w;
    int len = vmax;
    if (fo & 2) len = shorten_window(sm, cs, te, nok, vmax, status);
    const bool fast = fo != 0;  // a shortened window counts as fast-decaying
    if (fast || t0 + len >= L) {  // the extra terms
        if (!scan_extra<kPro>(sm, cs, te, len, fast, t0 + len >= L, abort_flag, status))
            return false;
    }
    if (te == 0) {
        win[cs & (kWinRing - 1)] = make_int4(t0, len, fast ? 1 : 0, 0);
        mbar_arrive(&bars[B_SCAN0 + (cs & 1)]);
    }
    return true;
}

__device__ __noinline__ int decay_scan(unsigned char* sm, int cs, int L, int te,
                                       volatile int* abort_flag, int* status) {
    return decay_scan_body<false>(sm, cs, L, te, abort_flag, status, 0.f, 0.f, 0.f);
}
__device__ __noinline__ int decay_scan_pro(unsigned char* sm, int cs, int L, int te,
                                           volatile int* abort_flag, int* status, float dt,
                                           float a, float lb) {
    return decay_scan_body<true>(sm, cs, L, te, abort_flag, status, dt, a, lb);
}
__device__ __noinline__ bool scan_rare(unsigned char* sm, int cs, int L, int te,
                                       volatile int* abort_flag, int* status) {
    return scan_rare_body<false>(sm, cs, L, te, abort_flag, status);
}
__device__ __noinline__ bool scan_rare_pro(unsigned char* sm, int cs, int L, int te,
                                           volatile int* abort_flag, int* status) {
    return scan_rare_body<true>(sm, cs, L, te, abort_flag, status);
}

// Self-test of the bounded waits: one CTA waits, through the kernels' own helper, on a barrier
// phase that nothing completes.  After kWaitLimit cycles (about 2 s) the wait gives up, records
// KDA_ERR_TIMEOUT in the status word and returns; the CTA holds no TMEM and issues no copies or
// MMAs, so it exits cleanly and the context stays usable.
__global__ void kda_wait_selftest_kernel(int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (wait_bar(&bar, 0, &abort_flag, status) && threadIdx.x == 0)
        report_status(status, KDA_ERR_INVALID_ARG);  // the phase cannot complete: never reached
}

// kCkpt: the variant that also writes state checkpoints; kPro: the variant that takes raw
// projections and runs the input prologue on the tiles as they arrive (the plain kernel carries
// no trace of either).
template <bool kCkpt, bool kPro>
__global__ void __launch_bounds__(kThreadsTC, 1)
kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g, const TcParams p,
                      const __grid_constant__ SeqOrder order) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int H = p.H;
    // blockIdx.x = rank * H + head: all heads of the longest sequence dispatch first
    const int rank = (int)(blockIdx.x / (unsigned)H);
    const int h = (int)(blockIdx.x % (unsigned)H);
    const int n = rank < order.count ? (int)order.seq[rank] : rank;
    const int64_t seq_begin = p.cu_seqlens[n];
    const int64_t seq_len = p.cu_seqlens[n + 1] - seq_begin;
    const int64_t unit = (int64_t)n * H + h;
    const SegPlan sp = segment_plan(seq_len, H);
    const int nseg = sp.nseg;
    // the device cu_seqlens must agree with the host plan the buffers were sized from
    bool bad = seq_begin < 0 || seq_len < 0 || seq_begin + seq_len > order.total_tokens ||
               (order.count > 0 && seq_len != order.len[n]);

    // ---- work item of this CTA ----
    int item;
    int sigma = 0;
    if (p.pass == 0) {
        if (nseg == 1) {
            if (blockIdx.z != 0) return;
            item = ITEM_WHOLE;
        } else {
            sigma = blockIdx.z >> 1;
            if (sigma >= nseg - 1) return;
            item = (blockIdx.z & 1) ? ITEM_TRANS : ITEM_TILDE;
        }
    } else {
        if (nseg == 1 || (int)blockIdx.z >= nseg) return;
        sigma = blockIdx.z;
        item = ITEM_SEGMENT;
    }
    const int64_t seg_tokens = (int64_t)sp.seg_chunks * kChunk;
    const int64_t seq0 = item == ITEM_WHOLE ? seq_begin : seq_begin + sigma * seg_tokens;
    const int L = (int)(item == ITEM_WHOLE ? seq_len : min(seg_tokens, seq_len - sigma * seg_tokens));
    int64_t slot = 0;  // workspace slot of (sequence, segment)
    if (item != ITEM_WHOLE) {
        int64_t base = 0;
        for (int m = 0; m < n; ++m) {
            const int ns = segment_plan((int64_t)p.cu_seqlens[m + 1] - p.cu_seqlens[m], H).nseg;
            if (ns > 1) base += ns;
        }
        bad |= base + nseg > order.total_slots;
        slot = ((base + sigma) * H + h) * (int64_t)(kDim * kDim);
    }
    if (kCkpt && p.ckpt && !bad) {  // the checkpoints this sequence writes fit the host's count
        const int every = kChunk * p.ckpt_chunks;
        int64_t base = 0;
        for (int m = 0; m <= n; ++m) base += (p.cu_seqlens[m + 1] - p.cu_seqlens[m]) / every;
        bad |= base > order.total_ckpts;
    }
    if (bad) {
        if (threadIdx.x == 0) report_status(p.status, KDA_ERR_INVALID_ARG);
        return;
    }
    const bool has_out = item == ITEM_WHOLE || item == ITEM_SEGMENT;
    const bool zero_v = item == ITEM_TRANS;
    const float* init_src = item == ITEM_WHOLE
                                ? (p.init_state ? p.init_state + unit * (kDim * kDim) : nullptr)
                                : (item == ITEM_SEGMENT ? p.ws_in + slot : nullptr);
    float* final_dst = item == ITEM_WHOLE ? (p.final_state ? p.final_state + unit * (kDim * kDim) : nullptr)
                       : item == ITEM_TILDE ? p.ws_tilde + slot
                       : item == ITEM_TRANS ? p.ws_trans + slot
                       : (sigma == nseg - 1 && p.final_state ? p.final_state + unit * (kDim * kDim)
                                                              : nullptr);

    if (L <= 0) {  // empty sequence: the final state is the initial state
        if (final_dst) {
            for (int e = tid; e < kDim * kDim; e += blockDim.x)
                final_dst[e] = init_src ? init_src[e] : 0.f;
        }
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 8);
    volatile int* kqg_issued = reinterpret_cast<volatile int*>(sm + OFF_MISC + 16);
    float* beta_s = reinterpret_cast<float*>(sm + OFF_BETA);
    float* er = reinterpret_cast<float*>(sm + OFF_ER);
    float* part = reinterpret_cast<float*>(sm + OFF_PART);
    float* gc_s = reinterpret_cast<float*>(sm + OFF_GC);
    float* sc = reinterpret_cast<float*>(sm + OFF_SC);
    const int4* win = reinterpret_cast<const int4*>(sm + OFF_WIN);
    // Chunk c covers tokens [t0, t0 + len) of this item, win[c % kWinRing] = {t0, len}, written by
    // the decay scan of chunk c before it releases the chunk (barrier B_SCAN).  win_end(c) is
    // where chunk c + 1 starts; there is a chunk c + 1 iff win_end(c) < L.
    auto win_end = [&](int c) {
        const int2 w = *reinterpret_cast<const int2*>(&win[c & (kWinRing - 1)]);
        return w.x + w.y;
    };
    auto win_start = [&](int c) { return c == 0 ? 0 : win_end(c - 1); };

    if (warp == kWarpTma) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    for (int e = tid; e < 2 * 8192 / 16; e += blockDim.x)
        reinterpret_cast<uint4*>(sm + OFF_TB0)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (zero_v)  // a transition item carries zero values: v stays zero, never loaded
        for (int e = tid; e < 16384 / 16; e += blockDim.x)
            reinterpret_cast<uint4*>(sm + OFF_V)[e] = make_uint4(0u, 0u, 0u, 0u);
    if (!has_out)  // no outputs: q is never loaded and its rows stay zero (Q_r unused)
        for (int e = tid; e < 4 * 8192 / 16; e += blockDim.x)
            reinterpret_cast<uint4*>(sm + ((e >> 10) ? OFF_KQW1 : OFF_KQW0) +
                                     ((e >> 9) & 1) * KQW_REGION + 8192)[e & 511] =
                make_uint4(0u, 0u, 0u, 0u);
    if (tid == 32) {
        for (int i = 0; i < B_COUNT; ++i)
            mbar_init(&bars[i], i == B_KQPRO0 || i == B_KQPRO1 ? kPrepThreads / 32 : 1);
        *abort_flag = 0;
        *kqg_issued = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t a_base = saddr(sm);
    // shared addresses of the per-slot tiles (slot s = chunk & 1)
    auto a_kq = [&](int s) { return a_base + (s ? OFF_KQW1 : OFF_KQW0); };
    auto kmh_off = [](int c) { const int s3 = c % 3; return s3 == 0 ? OFF_KMH0 : s3 == 1 ? OFF_KMH1 : OFF_KMH2; };
    auto a_kmh = [&](int c) { return a_base + kmh_off(c); };  // K_m slot of chunk c
    auto a_p = [&](int s) { return a_base + (s ? OFF_P1 : OFF_P0); };
    auto a_tb = [&](int s) { return a_base + (s ? OFF_TB1 : OFF_TB0); };
    // TMA issue helpers: k, q of chunk c into slot c & 1 (once M4 two chunks back has read the
    // slot), g of chunk c (once the factor pass of chunk c - 1 has read it), v of chunk c
    auto issue_kq = [&](int c) {
        const int s = c & 1;
        unsigned char* kq = sm + (s ? OFF_KQW1 : OFF_KQW0);
        uint64_t* full = &bars[B_FULL0 + s];
        const int t0 = (int)(seq0 + win_start(c));
        mbar_arrive_expect_tx(full, has_out ? 32768 : 16384);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(kq + r * KQW_REGION, &tm_k, full, 64 * r, h, t0);
            if (has_out)  // q only shapes outputs
                tma_load_3d(kq + r * KQW_REGION + 8192, &tm_q, full, 64 * r, h, t0);
        }
        *kqg_issued = c + 1;
    };
    auto issue_g = [&](int c) {
        uint64_t* full = &bars[B_GFULL];
        const int t0 = (int)(seq0 + win_start(c));
        mbar_arrive_expect_tx(full, 16384);
#pragma unroll
        for (int r = 0; r < 2; ++r) tma_load_3d(sm + OFF_G + r * 8192, &tm_g, full, 64 * r, h, t0);
    };
    auto issue_v = [&](int c) {
        if (zero_v) {
            mbar_arrive(&bars[B_VFULL]);
            return;
        }
        const int t0 = (int)(seq0 + win_start(c));
        mbar_arrive_expect_tx(&bars[B_VFULL], 16384);
        tma_load_3d(sm + OFF_V, &tm_v, &bars[B_VFULL], 0, h, t0);
        tma_load_3d(sm + OFF_V + 8192, &tm_v, &bars[B_VFULL], 64, h, t0);
    };

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ prep MMA issuer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_g);
            // k and q first: their copy count is published before the scan of chunk 0 can
            // start (the epilogue issues k and q of chunk 1 once chunk 0's window is known)
            issue_kq(0);
            issue_g(0);
            issue_v(0);
            int g_issued = 1;
            const uint32_t rP = tmem + T_P;
            const uint32_t a_v = saddr(sm + OFF_V);
            const uint32_t id_kk64 = idesc_bf16(128, 64, false, false);
            const uint32_t id_mk64 = idesc_bf16(128, 64, true, false);
            int v_issued = 1;
            // M1: [K_p ; Q_r] K_m^T of chunk c into the raw A / P tile
            auto issue_m1 = [&](const int c) -> bool {
                const int s = c & 1;
                if (!spin_bar(&bars[B_FACT0 + s], (c >> 1) & 1, abort_flag, p.status)) return false;
                // the factor pass and the scan have read g of chunk c: load g of chunk c + 1
                if (win_end(c) < L) {
                    issue_g(c + 1);
                    g_issued = c + 2;
                }
                tc_fence_after();
                const uint64_t dq = smem_desc(a_kq(s), 16, 1024);
                const uint64_t dh = smem_desc(a_kmh(c), 16, 1024);
#pragma unroll
                for (int j = 0; j < 8; ++j)  // 16 B descriptor units: K step 32 B
                    mma_ss(rP, dq + (j >> 2) * (KQW_REGION >> 4) + (j & 3) * 2,
                           dh + (j >> 2) * 512 + (j & 3) * 2, id_kk64, j > 0);
                mma_commit(&bars[B_AP0 + s]);
                return true;
            };
            for (int c = -1;; ++c) {  // M1 of chunk 0 first, then chunk by chunk
                if (c >= 0) {
                    const int s = c & 1;
                    // M2: W^T = K_p^T (T diag(beta))^T into the O^T columns of this chunk's block,
                    // once the epilogue has read that block two chunks ago.  (A per-slot barrier: a
                    // single one could run two phases ahead of this wait.)
                    if (!spin_bar(&bars[B_TB0 + s], (c >> 1) & 1, abort_flag, p.status)) break;
                    // M6 of chunk c - 1 (queued at the same moment) goes first: the factors of
                    // chunk c + 1 wait on it to free K_m, while W of chunk c is needed later
                    if (c >= 1 && !spin_bar(&bars[B_M6ISS], (c - 1) & 1, abort_flag, p.status)) break;
                    if (c >= 2 &&
                        !spin_bar(&bars[B_UFREE0 + s], ((c - 2) >> 1) & 1, abort_flag, p.status))
                        break;
                    tc_fence_after();
                    const uint32_t rX = tmem + (s ? T_X1 : T_X0);
                    {
                        const uint64_t da = smem_desc(a_kq(s), KQW_REGION, 1024);
                        const uint64_t db = smem_desc(a_tb(s), 16, 1024);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_ss(rX + 64, da + 128 * j, db + 2 * j, id_mk64, j > 0);
                    }
                    mma_commit(&bars[B_WDONE0 + s]);
                    // M3: U_bar^T = V^T (T diag(beta))^T into the U^T columns, once v has landed
                    // (and, for raw inputs, has been through Swish)
                    if (!spin_bar(&bars[kPro ? B_VPRO : B_VFULL], c & 1, abort_flag, p.status))
                        break;
                    tc_fence_after();
                    {
                        const uint64_t da = smem_desc(a_v, 8192, 1024);
                        const uint64_t db = smem_desc(a_tb(s), 16, 1024);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_ss(rX, da + 128 * j, db + 2 * j, id_mk64, j > 0);
                    }
                    mma_commit(&bars[B_VFREE0 + s]);
                    // the v buffer is free once M3 has read it: load the next chunk's v
                    if (win_end(c) >= L) break;  // chunk c was the last
                    if (!spin_bar(&bars[B_VFREE0 + s], (c >> 1) & 1, abort_flag, p.status))
                        break;
                    issue_v(c + 1);
                    v_issued = c + 2;
                }
                // the next chunk's factors follow this chunk's inverse
                if (!issue_m1(c + 1)) break;
            }
            mma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, kWaitLimit);
            if (*abort_flag) {  // let every issued copy land before the CTA can exit
                mbar_wait(&bars[B_VFULL], (v_issued - 1) & 1, kWaitLimit);
                const int nk = *kqg_issued;
                for (int c = nk - 2; c < nk; ++c)
                    if (c >= 0) mbar_wait(&bars[B_FULL0 + (c & 1)], (c >> 1) & 1, kWaitLimit);
                mbar_wait(&bars[B_GFULL], (g_issued - 1) & 1, kWaitLimit);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ serial MMA issuer
        if (lane == 0) {
            const uint32_t rS = tmem + T_S, rSA = tmem + T_SA;
            const uint32_t id_kk64 = idesc_bf16(128, 64, false, false);
            const uint32_t id_kk128 = idesc_bf16(128, 128, false, false);
            const uint32_t id_km128 = idesc_bf16(128, 128, false, true);
            for (int c = 0;; ++c) {
                const int s = c & 1;
                const uint32_t rX = tmem + (s ? T_X1 : T_X0);  // [U^T | O^T]
                // M4: [U^T | O^T] += X [-W ; Q_r]^T  (U^T starts at U_bar^T, O^T at zero)
                if (!spin_bar(&bars[B_WN0 + s], (c >> 1) & 1, abort_flag, p.status)) break;
                if (!spin_bar(&bars[B_SREADY], c & 1, abort_flag, p.status)) break;
                if (!spin_bar(&bars[B_VFREE0 + s], (c >> 1) & 1, abort_flag, p.status)) break;
                tc_fence_after();
                {
                    const uint64_t db = smem_desc(a_kq(s), 16, 1024);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        mma_ts(rX, rSA + 8 * j, db + (j >> 2) * (KQW_REGION >> 4) + (j & 3) * 2,
                               id_kk128, 1);
                }
                mma_commit(&bars[B_XDONE]);
                // M6 + M5: X += U^T K_m (2 split terms), O^T += U^T P^T (3 split terms);
                // U^T hi / lo sit in place of U^T (cols 0-31 / 32-63 of this chunk's block)
                if (!spin_bar(&bars[B_UREADY], c & 1, abort_flag, p.status)) break;
                const bool more = win_end(c) < L;
                // keep these off the tensor pipe while chunk c+1's inverse uses mma.sync
                if (more &&
                    !spin_bar(&bars[B_TB0 + ((c + 1) & 1)], ((c + 1) >> 1) & 1, abort_flag, p.status))
                    break;
                tc_fence_after();
                {
                    const uint32_t rUH = rX, rUL = rX + 32, rO = rX + 64;
                    const uint64_t dph = smem_desc(a_p(s), 16, 1024);
                    const uint64_t dpl = smem_desc(a_p(s) + 8192, 16, 1024);
                    const uint64_t dk = smem_desc(a_kmh(c), 8192, 1024);
                    // the state update first: the next chunk waits on it, the output does not
#pragma unroll
                    for (int j = 0; j < 4; ++j) mma_ts(rS, rUH + 8 * j, dk + 128 * j, id_km128, 1);
#pragma unroll
                    for (int j = 0; j < 4; ++j) mma_ts(rS, rUL + 8 * j, dk + 128 * j, id_km128, 1);
                    if (!more) {  // the final state: K_m's residue too (in the next K_m slot)
                        const uint64_t dkr = smem_desc(a_kmh(c + 1), 8192, 1024);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_ts(rS, rUH + 8 * j, dkr + 128 * j, id_km128, 1);
                    }
                    mma_commit(&bars[B_KMFREE0 + c % 3]);  // K_m of this slot has been read
                    mma_commit(&bars[B_SDONE]);
                    mbar_arrive(&bars[B_M6ISS]);  // M6 is queued: the next M2 may follow it
                    if (has_out) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_ts(rO, rUH + 8 * j, dph + 2 * j, id_kk64, 1);
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_ts(rO, rUL + 8 * j, dph + 2 * j, id_kk64, 1);
#pragma unroll
                        for (int j = 0; j < 4; ++j) mma_ts(rO, rUH + 8 * j, dpl + 2 * j, id_kk64, 1);
                    }
                }
                mma_commit(&bars[B_PFREE0 + s]);  // P of this slot has been read
                mma_commit(&bars[B_OSDONE]);
                if (!more) break;
            }
            // every issued MMA completes before TMEM can be released
            mma_commit(&bars[B_SPARE]);
            mbar_wait(&bars[B_SPARE], 0, kWaitLimit);
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------------ prep (warps 2-9)
        const int tp = tid - kWarpPrep0 * 32;
        const int cg = tp & 15;         // channel group of the factor pass
        const int tg = tp >> 4;         // token group of the factor pass
        const int c8 = 8 * cg;
        const int wp = warp - kWarpPrep0;
        const int q4 = warp & 3;
        const int colhalf = (warp - kWarpPrep0) >> 2;
        const int row_abs = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        float* Am = reinterpret_cast<float*>(sm + OFF_KML);
        const float* qk_s = reinterpret_cast<const float*>(sm + OFF_QK);
        // chunk c decays faster than kHeavyDecay in some channel (recorded by its scan)
        auto chunk_heavy = [&](int c) { return win[c & (kWinRing - 1)].z != 0; };
        const unsigned short* beta_u = reinterpret_cast<const unsigned short*>(p.beta) + seq0 * H + h;
        unsigned short beta_raw = 0;  // raw bf16 bits; converted one chunk after the load
        int beta_t0 = 0;              // item token where the rows in beta_raw start
        int t0_next = 0;              // first token of the next chunk to factor (its scan's)
        if (tp < min(kChunk, L)) beta_raw = beta_u[(int64_t)tp * H];
        // scratch of the inverse: the four blocks of the upper quadrant of A / T (rows 0-31,
        // columns 32-63), which no step stores or reads otherwise
        auto Yb = [&](int k) { return Am + (k >> 1) * 16 * LDA_T + 32 + (k & 1) * 16; };
        // beta of chunk c (two chunks are live: the next chunk's factors are made before this
        // chunk's W epilogue)
        auto beta_ring = [&](int c) { return beta_s + (c & 1) * kChunk; };
        // decay factors of chunk c (from its q, k, g tile)
        auto factor = [&](const int c) -> bool {
            const int s = c & 1;
            unsigned char* kq = sm + (s ? OFF_KQW1 : OFF_KQW0);
            unsigned char* kmh = sm + kmh_off(c);
            if (!wait_bar(&bars[B_FULL0 + s], (c >> 1) & 1, abort_flag, p.status)) return false;
            if constexpr (kPro) {
                // raw k, q -> Swish, row norm, bf16, in place.  This needs only the k / q tiles,
                // so it runs before the wait for the decay scan, off the serial chain.
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    const uint32_t o = sw128_offset(4 * tg + i, c8, KQW_ROWS);
                    float kv[8], qv[8];
                    unpack8(*reinterpret_cast<const uint4*>(kq + o), kv);
                    unpack8(*reinterpret_cast<const uint4*>(kq + o + 64 * 128), qv);
                    pro_swish_l2_kq(kv, qv, p.pro_q_scale);  // packing rounds them to bf16
                    *reinterpret_cast<uint4*>(kq + o) = pack8(kv);
                    *reinterpret_cast<uint4*>(kq + o + 64 * 128) = pack8(qv);
                }
                __syncwarp();  // the scan may read the transformed tiles
                if (lane == 0) mbar_arrive(&bars[B_KQPRO0 + s]);
            }

            // ---- decay factors: thread (tg, cg) owns tokens 4tg..4tg+3, channels 8cg..8cg+7.
            // The window, the token-group prefixes of g, G_C and e^{r} come from the epilogue
            // warps' scan.
            if (tp < kChunk) {
                // beta of the rest of the 64-token block from the chunk's first token (its window
                // length is not known yet), prefetched one chunk ago for the block start; a chunk
                // that starts inside a block (after a shortened window) loads it now
                const int t0c = t0_next;  // where chunk c - 1's window ended
                const int vm = min(L - t0c, kChunk - (t0c & (kChunk - 1)));
                if (beta_t0 != t0c) beta_raw = tp < vm ? beta_u[((int64_t)t0c + tp) * H] : 0;
                float bt = __uint_as_float((uint32_t)beta_raw << 16);
                if constexpr (kPro) bt = tp < vm ? round_bf16(pro_sigmoid(bt)) : 0.f;
                beta_ring(c)[tp] = bt;
                // fetch the next block's beta now; it is needed one chunk later
                const int tn = (t0c & ~(kChunk - 1)) + kChunk;
                const int vn = min(L - tn, kChunk);
                beta_raw = tp < vn ? beta_u[((int64_t)tn + tp) * H] : 0;
                beta_t0 = tn;
            }
            // g has landed (the scan waited for it too) and its prefixes are in place
            if (!wait_bar(&bars[B_GFULL], c & 1, abort_flag, p.status) ||
                !wait_bar(&bars[B_SCAN0 + s], (c >> 1) & 1, abort_flag, p.status))
                return false;
            const int2 wc = *reinterpret_cast<const int2*>(&win[c & (kWinRing - 1)]);
            const int valid = wc.y;  // rows past the window are padding
            t0_next = wc.x + wc.y;
            if (tp < kChunk && tp >= valid) beta_ring(c)[tp] = 0.f;
            {
                float G[8], r[8];
                {
                    const float4 a = *reinterpret_cast<const float4*>(part + tg * kDim + c8);
                    const float4 b = *reinterpret_cast<const float4*>(part + tg * kDim + c8 + 4);
                    const float4 ga = *reinterpret_cast<const float4*>(gc_s + c8);
                    const float4 gb = *reinterpret_cast<const float4*>(gc_s + c8 + 4);
                    // G - r in log2 units (the factors are exp2 of it), from the exclusive prefix
                    const float hl = 0.5f * kLog2eTC;
                    r[0] = hl * ga.x; r[1] = hl * ga.y; r[2] = hl * ga.z; r[3] = hl * ga.w;
                    r[4] = hl * gb.x; r[5] = hl * gb.y; r[6] = hl * gb.z; r[7] = hl * gb.w;
                    G[0] = fmaf(a.x, kLog2eTC, -r[0]); G[1] = fmaf(a.y, kLog2eTC, -r[1]);
                    G[2] = fmaf(a.z, kLog2eTC, -r[2]); G[3] = fmaf(a.w, kLog2eTC, -r[3]);
                    G[4] = fmaf(b.x, kLog2eTC, -r[4]); G[5] = fmaf(b.y, kLog2eTC, -r[5]);
                    G[6] = fmaf(b.z, kLog2eTC, -r[6]); G[7] = fmaf(b.w, kLog2eTC, -r[7]);
                }
                // K_m of this slot is overwritten only after M6 three chunks back has read it
                if (c >= 3 && !wait_bar(&bars[B_KMFREE0 + c % 3], ((c - 3) / 3) & 1, abort_flag,
                                        p.status))
                    return false;
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    // one token per step: rows t and 64 + t of the slot tile (k, q; they share the
                    // swizzle phase t & 7, so one offset serves both, and they are replaced in
                    // place by K_p, Q_r) and row t of the g buffer
                    const int t = 4 * tg + i;
                    const uint32_t o = sw128_offset(t, c8, KQW_ROWS);
                    uint4 gr = make_uint4(0u, 0u, 0u, 0u);
                    if (t < valid)
                        gr = *reinterpret_cast<const uint4*>(sm + OFF_G + sw128_offset(t, c8, 64));
                    const uint4 kr = *reinterpret_cast<const uint4*>(kq + o);
                    const uint4 qr4 = *reinterpret_cast<const uint4*>(kq + o + 64 * 128);
                    float gv[8], kv[8], qv[8];
                    unpack8(gr, gv);
                    unpack8(kr, kv);
                    unpack8(qr4, qv);
                    float kp[8], qr[8], km[8];
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        const float2 g2 = fma_f32x2(make_float2(gv[j], gv[j + 1]),
                                                    make_float2(kLog2eTC, kLog2eTC),
                                                    make_float2(G[j], G[j + 1]));
                        G[j] = g2.x;  // G - r, log2 units
                        G[j + 1] = g2.y;
                        const float2 e = make_float2(ex2_approx(G[j]), ex2_approx(G[j + 1]));
                        const float2 ei = make_float2(ex2_approx(-G[j]), ex2_approx(-G[j + 1]));
                        const float2 k2 = make_float2(kv[j], kv[j + 1]);
                        const float2 a = mul_f32x2(k2, e);
                        const float2 b = mul_f32x2(make_float2(qv[j], qv[j + 1]), e);
                        const float2 m = mul_f32x2(k2, ei);
                        kp[j] = a.x; kp[j + 1] = a.y;
                        qr[j] = b.x; qr[j + 1] = b.y;
                        km[j] = m.x; km[j + 1] = m.y;
                    }
                    *reinterpret_cast<uint4*>(kq + o) = pack8(kp);
                    *reinterpret_cast<uint4*>(kq + o + 64 * 128) = pack8(qr);
                    *reinterpret_cast<uint4*>(kmh + sw128_offset(t, c8, 64)) = pack8(km);
                }
            }
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_FACT0 + s]);
            return true;
        };
        // A and P of chunk c from TMEM
        auto ap_epilogue = [&](const int c) -> bool {
            const int s = c & 1;
            unsigned char* pt = sm + (s ? OFF_P1 : OFF_P0);
            // ---- A (rows 0-63) and P (rows 64-127) from TMEM ----
            if (!wait_bar(&bars[B_AP0 + s], (c >> 1) & 1, abort_flag, p.status)) return false;
            if (c >= 2 &&
                !wait_bar(&bars[B_PFREE0 + s], ((c - 2) >> 1) & 1, abort_flag, p.status))
                return false;
            tc_fence_after();
            {
                uint32_t v[32];
                tmem_ld32(tmem + T_P + 32 * colhalf + lane_off, v);
                if (row_abs < kChunk) {
                    const int t = row_abs;
                    const float bt = beta_ring(c)[t];
                    // only the strictly lower triangle is ever read, so it is stored unmasked;
                    // the upper quadrant (rows 0-31, columns 32-63) is the inverse's scratch
                    if (colhalf <= q4) {
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            float4 o;
                            const int col = 32 * colhalf + 4 * j4;
                            o.x = bt * __uint_as_float(v[4 * j4 + 0]);
                            o.y = bt * __uint_as_float(v[4 * j4 + 1]);
                            o.z = bt * __uint_as_float(v[4 * j4 + 2]);
                            o.w = bt * __uint_as_float(v[4 * j4 + 3]);
                            *reinterpret_cast<float4*>(Am + t * LDA_T + col) = o;
                        }
                    }
                    // ---- T = (I + A)^{-1}, diagonal 16 x 16 blocks by forward substitution.
                    // The warp that stored a diagonal 32 x 32 quadrant of A inverts its two
                    // blocks right away (16 lanes per block, one column each) while the other
                    // warps are still on P.
                    if (q4 == colhalf) {
                        __syncwarp();
                        const int b = 2 * q4 + (lane >> 4), col = lane & 15;
                        const float* Ab = Am + (16 * b) * LDA_T + 16 * b;
                        float x[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {  // four partial sums shorten the chain
                            float s4[4] = {(i == col) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int q = 0; 4 * q < i; ++q) {  // row i, four entries at a time
                                const float4 a4 =
                                    *reinterpret_cast<const float4*>(Ab + i * LDA_T + 4 * q);
                                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    if (4 * q + u < i) s4[u] = fmaf(-av[u], x[4 * q + u], s4[u]);
                            }
                            x[i] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                        }
                        __syncwarp();
                        float* Tb = Am + (16 * b) * LDA_T + 16 * b;
#pragma unroll
                        for (int i = 0; i < 16; ++i) Tb[i * LDA_T + col] = x[i];
                    }
                } else if (has_out) {  // P only shapes outputs
                    const int t = row_abs - kChunk;
#pragma unroll
                    for (int j8 = 0; j8 < 4; ++j8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int col = 32 * colhalf + 8 * j8 + 2 * u;
                            const float x0 = col <= t ? __uint_as_float(v[8 * j8 + 2 * u]) : 0.f;
                            const float x1 = col + 1 <= t ? __uint_as_float(v[8 * j8 + 2 * u + 1]) : 0.f;
                            const uint32_t hh = pack_bf16(x0, x1);
                            hi[u] = hh;
                            lo[u] = pack_bf16(x0 - __uint_as_float(hh << 16),
                                              x1 - __uint_as_float(hh & 0xffff0000u));
                        }
                        const uint32_t off = sw128_offset(t, 32 * colhalf + 8 * j8, 64);
                        *reinterpret_cast<uint4*>(pt + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(pt + 8192 + off) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    if (colhalf == (t >> 5) && chunk_heavy(c)) {  // it stored P[t][t]: use q_t . k_t
                        const float qkt = qk_s[(c & 3) * kChunk + t];
                        const uint32_t hh = pack_bf16(qkt, 0.f);
                        const uint32_t ll = pack_bf16(qkt - __uint_as_float(hh << 16), 0.f);
                        uint32_t* ph = reinterpret_cast<uint32_t*>(
                            pt + sw128_offset(t, t & ~7, 64) + ((t & 7) >> 1) * 4);
                        uint32_t* pl = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(ph) + 8192);
                        if (t & 1) {  // the high half of the pair (t - 1, t)
                            *ph = (*ph & 0xffffu) | (hh << 16);
                            *pl = (*pl & 0xffffu) | (ll << 16);
                        } else {      // the low half of (t, t + 1); column t + 1 is zero
                            *ph = hh;
                            *pl = ll;
                        }
                    }
                }
            }
            tc_fence_before();
            named_bar(kBarPrep, kPrepThreads);
            return true;
        };
        // T diag(beta) of chunk c
        auto inverse = [&](const int c) -> void {
            const int s = c & 1;
            unsigned char* tb = sm + (s ? OFF_TB1 : OFF_TB0);
            // ---- off-diagonal blocks on the tensor cores (tf32), with D = blockdiag(T_II) and
            //      N = D A_off (block-nilpotent):  T = (I - N + N^2 - N^3) D ----
            if (wp < 6) {  // N_IJ = T_II A_IJ, in place of A_IJ
                const int I = pair_i(wp), J = pair_j(wp);
                float acc[2][4];
                block_product(acc, Am + (16 * I) * LDA_T + 16 * I, LDA_T, 1.f, nullptr, 0,
                              Am + (16 * I) * LDA_T + 16 * J, LDA_T, lane);
                __syncwarp();
                store_block(Am + (16 * I) * LDA_T + 16 * J, LDA_T, acc, lane);
            }
            named_bar(kBarPrep, kPrepThreads);
            if (wp < 3) {  // N^2_20, N^2_31 (then N^3_30 = N^2_31 N_10), N^2_30
                // wp 0: N^2_20 = N_21 N_10;  wp 1: N^2_31 = N_32 N_21, then N^3_30 = N^2_31 N_10;
                // wp 2: N^2_30 = N_31 N_10 + N_32 N_20.  One code path, operands picked per warp.
                float acc[2][4];
                block_product(acc,
                              Am + (wp == 0 ? 32 * LDA_T + 16 : wp == 1 ? 48 * LDA_T + 32 : 48 * LDA_T + 16),
                              LDA_T, 1.f, nullptr, nullptr,
                              Am + (wp == 1 ? 32 * LDA_T + 16 : 16 * LDA_T), LDA_T, lane);
                if (wp != 0) {
                    if (wp == 1) {
                        store_block(Yb(1), LDA_T, acc, lane);
                        __syncwarp();
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
                            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
                    }
                    block_mma(acc, wp == 1 ? Yb(1) : Am + 48 * LDA_T + 32, LDA_T,
                              1.f, nullptr, nullptr, Am + (wp == 1 ? 16 * LDA_T : 32 * LDA_T), LDA_T,
                              lane);
                }
                store_block(Yb(wp == 0 ? 0 : wp == 1 ? 3 : 2), LDA_T, acc, lane);
            }
            named_bar(kBarPrep, kPrepThreads);
            if (wp < 6) {  // T_IJ = C_IJ T_JJ with C = -N + N^2 - N^3 (block by block)
                const int I = pair_i(wp), J = pair_j(wp);
                const float* n2 = (I == 2 && J == 0) ? Yb(0) : (I == 3 && J == 1) ? Yb(1)
                                : (I == 3 && J == 0) ? Yb(2) : nullptr;
                const float* n3 = (I == 3 && J == 0) ? Yb(3) : nullptr;
                float acc[2][4];
                block_product(acc, Am + (16 * I) * LDA_T + 16 * J, LDA_T, -1.f, n2, n3,
                              Am + (16 * J) * LDA_T + 16 * J, LDA_T, lane);
                store_block_tb(tb, I, J, acc, beta_ring(c), lane);
            } else {  // the diagonal blocks T_II, two per warp, into the bf16 operand tile
                const int g = lane >> 2, tq = lane & 3;
#pragma unroll 1
                for (int I = 2 * (wp - 6); I < 2 * (wp - 6) + 2; ++I) {
                    const float* Tb = Am + 16 * I * (LDA_T + 1);
                    float acc[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float2 u = *reinterpret_cast<const float2*>(Tb + g * LDA_T + 8 * nt + 2 * tq);
                        const float2 w =
                            *reinterpret_cast<const float2*>(Tb + (g + 8) * LDA_T + 8 * nt + 2 * tq);
                        acc[nt][0] = u.x; acc[nt][1] = u.y; acc[nt][2] = w.x; acc[nt][3] = w.y;
                    }
                    store_block_tb(tb, I, I, acc, beta_ring(c), lane);
                }
            }
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_TB0 + s]);
        };
        // -W of chunk c into its slot tile
        auto w_epilogue = [&](const int c) -> bool {
            const int s = c & 1;
            unsigned char* kq = sm + (s ? OFF_KQW1 : OFF_KQW0);
            // ---- -W into rows 0-63 of the slot tile (K-major [t][c]), over K_p ----
            if (!wait_bar(&bars[B_WDONE0 + s], (c >> 1) & 1, abort_flag, p.status)) return false;
            tc_fence_after();
            {
                uint32_t v[32];
                const uint32_t rW = tmem + (s ? T_X1 : T_X0) + 64 + 32 * colhalf + lane_off;
                tmem_ld32(rW, v);  // W^T[c = row_abs][t]
                // Lanes 2i and 2i+1 hold channels ch0 and ch0+1.  Each packs its own tokens
                // (j, j+4) and the two swap words: the even lane stores the low halves (token j),
                // the odd lane the high halves (token j+4), each as the bf16 pair (ch0, ch0+1).
                // Rows four apart put the two half-warps on disjoint banks of the swizzled tile.
                const bool odd = lane & 1;
                const uint32_t sel = odd ? 0x3276u : 0x5410u;
                // Rows t0 + j with j & 7 in 0..3 have swizzle phase (t0 + (j & 3)) & 7, so four
                // row bases per thread serve every store, plus a compile-time row offset.
                const int t0 = 32 * colhalf + (odd ? 4 : 0);
                unsigned char* wb[4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    wb[m] = kq + sw128_offset(t0 + m, row_abs & ~1, KQW_ROWS) - m * 128;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = (jj & 3) + 8 * (jj >> 2);
                    const uint32_t mine =
                        pack_bf16(-__uint_as_float(v[j]), -__uint_as_float(v[j + 4]));
                    const uint32_t partner = __shfl_xor_sync(0xffffffffu, mine, 1);
                    *reinterpret_cast<uint32_t*>(wb[j & 3] + j * 128) = __byte_perm(mine, partner, sel);
                }
                tmem_st32_zero(rW);  // O^T of this chunk accumulates from zero in M4
                tmem_st_wait();
            }
            tc_fence_before();
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_WN0 + s]);
            return true;
        };
        // Software pipeline: the W epilogue of chunk c-1 runs while the tensor core forms A and P
        // of chunk c, and the factors of chunk c+1 while it forms W of chunk c.
        // Each phase has a single call site (the lambdas are inlined where they are called).
        // kPro: Swish on v of chunk c in place before M3 of chunk c reads it
        auto v_prologue = [&](const int c) -> bool {
            if (!wait_bar(&bars[B_VFULL], c & 1, abort_flag, p.status)) return false;
            if (!zero_v) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4* src = reinterpret_cast<uint4*>(sm + OFF_V) + tp + kPrepThreads * j;
                    float x[8];
                    unpack8(*src, x);
                    pro_swish8(x);
                    *src = pack8(x);
                }
            }
            fence_async_shared();
            named_bar(kBarPrep, kPrepThreads);
            if (tp == 0) mbar_arrive(&bars[B_VPRO]);
            return true;
        };
        bool cur = false;  // chunk c exists
        for (int c = -1;; ++c) {
            if (c >= 1 && !w_epilogue(c - 1)) break;
            if (c >= 0) {
                if (!cur) break;  // the W epilogue of the last chunk was the final step
                if (!ap_epilogue(c)) break;
                inverse(c);
                if constexpr (kPro) {
                    if (!v_prologue(c)) break;
                }
            }
            // chunk c's window is known: factor(c) waited for its scan
            const bool next = c < 0 || win_end(c) < L;
            if (next && !factor(c + 1)) break;
            cur = next;
        }
    } else {
        // ------------------------------------------------------------ serial epilogue
        const int te = tid - kWarpEpi0 * 32;
        const int q4 = warp & 3;
        const int vch = 32 * q4 + lane;  // value channel = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        // state checkpoints (items with outputs only): this (sequence, head)'s first checkpoint
        // slot, and the sequence chunk of this item's chunk 0
        float* ckpt0 = nullptr;
        if (kCkpt && p.ckpt && has_out) {
            const int every = kChunk * p.ckpt_chunks;  // token offsets are int32
            int64_t base = 0;
#pragma unroll 1
            for (int m = 0; m < n; ++m) base += (p.cu_seqlens[m + 1] - p.cu_seqlens[m]) / every;
            ckpt0 = p.ckpt + (base * H + h) * (int64_t)(kDim * kDim);
        }
        const int chunk0 = item == ITEM_SEGMENT ? sigma * sp.seg_chunks : 0;
        float pro_dt = 0.f, pro_a = 0.f, pro_lb = 0.f;
        if constexpr (kPro) {
            pro_dt = p.pro_dt_bias ? p.pro_dt_bias[h * kDim + te] : 0.f;
            pro_a = pro_gate_rate(p.pro_A_log, h);
            pro_lb = p.pro_lb;
        }
        auto scan = [&](const int cs) -> bool {
            const int r = kPro ? decay_scan_pro(sm, cs, L, te, abort_flag, p.status, pro_dt,
                                                pro_a, pro_lb)
                               : decay_scan(sm, cs, L, te, abort_flag, p.status);
            if (r <= 0) return r == 0;
            return kPro ? scan_rare_pro(sm, cs, L, te, abort_flag, p.status)
                        : scan_rare(sm, cs, L, te, abort_flag, p.status);
        };
        bool ok = true;
        // c = -2 and -1 only scan chunks 0 and 1 (and set up X_0): one code path for the scan.
        // Chunk c + 1 exists iff win_end(c) < L, known once chunk c's scan is done (two chunks
        // ahead of this loop).
        for (int c = -2; ok; ++c) {
            const uint32_t rX = tmem + ((c & 1) ? T_X1 : T_X0) + lane_off;
            if (c == -1) {  // X_0 = S0^T diag(e^{r_0}); S0 = 0, I (transition items) or given
                const float* e0 = er;
                const float* s0 = init_src;
                for (int cc = 0; cc < kDim; cc += 32) {
                    uint32_t x[32], xb[16];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float sv = s0 ? s0[(cc + j) * kDim + vch]
                                            : (item == ITEM_TRANS && cc + j == vch ? 1.f : 0.f);
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
                // chunk 1 reuses the prefix array once the prep warps have read chunk 0's
                if (win_end(0) < L && !(ok = wait_bar(&bars[B_FACT0], 0, abort_flag, p.status)))
                    break;
            }
            if (c >= 0) {
                // ---- E1: U^T -> bf16 hi/lo A operands ----
                if (!(ok = wait_bar(&bars[B_XDONE], c & 1, abort_flag, p.status))) break;
                tc_fence_after();
                // M1, M2 and now M4 have read this slot's K_p / Q_r / -W rows: refill k and q with
                // chunk c + 2 (g was refilled after the factor pass; K_m is guarded by B_KMFREE)
                if (te == 0 && win_end(c) < L && win_end(c + 1) < L) issue_kq(c + 2);
                {
                    // read all 64 columns of U^T before writing hi / lo over them
                    uint32_t u[64], lo[32];
                    tmem_ld64(rX, u);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float x0 = __uint_as_float(u[2 * j]), x1 = __uint_as_float(u[2 * j + 1]);
                        const uint32_t hi = pack_bf16(x0, x1);
                        lo[j] = pack_bf16(x0 - __uint_as_float(hi << 16),
                                          x1 - __uint_as_float(hi & 0xffff0000u));
                        u[j] = hi;  // u[2j], u[2j+1] are consumed; slot j <= 2j is free
                    }
                    uint32_t hi32[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) hi32[j] = u[j];
                    tmem_st32(rX, hi32);
                    tmem_st32(rX + 32, lo);
                }
                tmem_st_wait();
                tc_fence_before();
                named_bar(kBarEpi, kEpiThreads);
                if (te == 0) mbar_arrive(&bars[B_UREADY]);
            }
            // The cumulative decay of chunk c + 2 (its g landed a chunk ago).  The prep warps
            // read chunk c + 1's prefixes before the W epilogue of chunk c, so before XDONE of
            // chunk c.
            const bool scan_next = c == -2 || ((c < 0 || win_end(c) < L) && win_end(c + 1) < L);
            if (scan_next && !(ok = scan(c + 2))) break;
            // k and q of chunk 1, once chunk 0's window has fixed where chunk 1 starts
            if (c == -2 && te == 0 && win_end(0) < L) issue_kq(1);
            if (c < 0) continue;

            // ---- E2: state rescale first (the next chunk's M4 waits on it), then O to HBM ----
            if (!(ok = wait_bar(&bars[B_SDONE], c & 1, abort_flag, p.status))) break;
            tc_fence_after();
            const int2 wc = *reinterpret_cast<const int2*>(&win[c & (kWinRing - 1)]);
            const int valid = wc.y;
            const int64_t tok0 = seq0 + wc.x;
            const bool last = wc.x + wc.y >= L;
            // The state after this chunk is a checkpoint when its window ends on a 64-token
            // block whose sequence position is a multiple of the interval (a ragged last chunk
            // never is).  S = X diag(e^{r_c}), transposed back, exactly as the final state.
            const int pos = wc.x + wc.y;
            const int done = chunk0 + pos / kChunk;
            float* ckd = (kCkpt && ckpt0 && (pos & (kChunk - 1)) == 0 && done % p.ckpt_chunks == 0)
                             ? ckpt0 + (int64_t)(done / p.ckpt_chunks - 1) * H * (kDim * kDim)
                             : nullptr;
            const float* ec = er + (c & 3) * kDim;
            if (ckd) store_state(ckd, tmem + T_S + lane_off, ec, vch);
            if (!last) {  // the scale of chunk c + 1 is from this warp group's own scan
                const float* scn = sc + ((c + 1) & 3) * kDim;
#pragma unroll 1
                for (int cc = 0; cc < kDim; cc += 32) {
                    uint32_t x[32], xb[16];
                    tmem_ld32(tmem + T_S + cc + lane_off, x);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 f = *reinterpret_cast<const float4*>(scn + cc + j);
                        x[j] = __float_as_uint(__uint_as_float(x[j]) * f.x);
                        x[j + 1] = __float_as_uint(__uint_as_float(x[j + 1]) * f.y);
                        x[j + 2] = __float_as_uint(__uint_as_float(x[j + 2]) * f.z);
                        x[j + 3] = __float_as_uint(__uint_as_float(x[j + 3]) * f.w);
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
            } else if (final_dst) {
                store_state(final_dst, tmem + T_S + lane_off, ec, vch);
            }
            if (!(ok = wait_bar(&bars[B_OSDONE], c & 1, abort_flag, p.status))) break;
            tc_fence_after();
            {
                if (has_out) {
                    // lanes 2i and 2i+1 (channels e, e+1) swap their packed token pairs so that
                    // the even lane stores token t and the odd lane token t+1 as a bf16 pair
                    const bool odd = lane & 1;
                    const uint32_t sel = odd ? 0x3276u : 0x5410u;  // as in the W epilogue
                    const int64_t tstride = (int64_t)H * kDim;
                    bf16* op = p.out + ((tok0 + (odd ? 1 : 0)) * H + h) * kDim + (vch & ~1);
#pragma unroll 1
                    for (int t0 = 0; t0 < 64; t0 += 16) {
                        uint32_t o[16];
                        tmem_ld16(rX + 64 + t0, o);
#pragma unroll
                        for (int t = 0; t < 16; t += 2) {
                            const uint32_t mine =
                                pack_bf16(__uint_as_float(o[t]), __uint_as_float(o[t + 1]));
                            const uint32_t partner = __shfl_xor_sync(0xffffffffu, mine, 1);
                            if (t0 + t + (odd ? 1 : 0) < valid)
                                *reinterpret_cast<uint32_t*>(op) = __byte_perm(mine, partner, sel);
                            op += 2 * tstride;
                        }
                    }
                }
                if (!last) {  // the block is free for chunk c + 2
                    tc_fence_before();
                    named_bar(kBarEpi, kEpiThreads);
                    if (te == 0) mbar_arrive(&bars[B_UFREE0 + (c & 1)]);
                }
            }
            if (last) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpTma) tmem_dealloc(tmem, 512);
}

// Composition of segment effects:
//   S_in(0) = initial state;  S_in(s+1) = M_s S_in(s) + S~_s
// ("k3_training_and_infra_notes", section 4.1: a segment's transition is evaluated without the
// incoming state and composed exactly afterwards).  fp32 on the CUDA cores; every S_in(s) is
// written to the workspace for the second pass.  The value channels (columns of S) evolve
// independently, so each split (sequence, head) runs as kCombineColBlocks CTAs, one per block of
// 16 columns, which spreads the serial chain over many SMs.
constexpr int kCombineThreads = 256;
constexpr int kCombineColBlocks = 8;
constexpr int kCombineCols = kDim / kCombineColBlocks;  // 16
constexpr int kCombineLdM = kDim + 2;  // M is kept transposed, rows padded against bank conflicts
__global__ void __launch_bounds__(kCombineThreads, 1)
kda_segment_combine_kernel(const int32_t* __restrict__ cu_seqlens, const float* __restrict__ init_state,
                           const float* __restrict__ ws_tilde, const float* __restrict__ ws_trans,
                           float* __restrict__ ws_in, int H, int* status,
                           const __grid_constant__ SeqOrder plan) {
    extern __shared__ __align__(16) float cs[];
    float* Mt = cs;                         // [128][130]: Mt[k][row] = M[row][k]
    float* S = cs + kDim * kCombineLdM;     // [128][16]: columns 16 cb .. 16 cb + 15 of the state
    const int n = blockIdx.x, h = blockIdx.y, cb = blockIdx.z, tid = threadIdx.x;
    const int64_t len = (int64_t)cu_seqlens[n + 1] - cu_seqlens[n];
    const int nseg = segment_plan(len, H).nseg;
    if (nseg <= 1) return;
    int64_t base = 0;
    for (int m = 0; m < n; ++m) {
        const int ns = segment_plan((int64_t)cu_seqlens[m + 1] - cu_seqlens[m], H).nseg;
        if (ns > 1) base += ns;
    }
    // the device cu_seqlens must agree with the host plan the workspace was sized from
    if (base + nseg > plan.total_slots || (plan.count > 0 && len != plan.len[n])) {
        if (tid == 0) report_status(status, KDA_ERR_INVALID_ARG);
        return;
    }
    const int64_t unit = (int64_t)n * H + h;
    const int c0 = kCombineCols * cb;
    // element e of the slice (4 floats): row e >> 2, columns c0 + 4 (e & 3) ..
    auto slice = [&](int e) { return (e >> 2) * kDim + c0 + 4 * (e & 3); };
    const float* s0 = init_state ? init_state + unit * (kDim * kDim) : nullptr;
    for (int e = tid; e < kDim * kCombineCols / 4; e += kCombineThreads)
        reinterpret_cast<float4*>(S)[e] =
            s0 ? *reinterpret_cast<const float4*>(s0 + slice(e)) : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const int r = 2 * (tid >> 2), cc = 4 * (tid & 3);  // rows r, r + 1; slice columns cc .. cc + 3
    for (int sg = 0; sg < nseg; ++sg) {
        const int64_t off = ((base + sg) * H + h) * (int64_t)(kDim * kDim);
        for (int e = tid; e < kDim * kCombineCols / 4; e += kCombineThreads)
            *reinterpret_cast<float4*>(ws_in + off + slice(e)) = reinterpret_cast<const float4*>(S)[e];
        if (sg == nseg - 1) break;
        for (int e = tid; e < kDim * kDim / 4; e += kCombineThreads) {
            const int row = e & (kDim - 1), k4 = 4 * (e >> 7);  // neighbouring lanes: rows
            const float4 v = *reinterpret_cast<const float4*>(ws_trans + off + row * kDim + k4);
            Mt[(k4 + 0) * kCombineLdM + row] = v.x;
            Mt[(k4 + 1) * kCombineLdM + row] = v.y;
            Mt[(k4 + 2) * kCombineLdM + row] = v.z;
            Mt[(k4 + 3) * kCombineLdM + row] = v.w;
        }
        __syncthreads();
        float acc[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < kDim; ++kk) {  // the same summation order for every element
            const float2 mm = *reinterpret_cast<const float2*>(Mt + kk * kCombineLdM + r);
            const float m0 = mm.x, m1 = mm.y;
            const float4 sv = *reinterpret_cast<const float4*>(S + kk * kCombineCols + cc);
            acc[0][0] = fmaf(m0, sv.x, acc[0][0]); acc[0][1] = fmaf(m0, sv.y, acc[0][1]);
            acc[0][2] = fmaf(m0, sv.z, acc[0][2]); acc[0][3] = fmaf(m0, sv.w, acc[0][3]);
            acc[1][0] = fmaf(m1, sv.x, acc[1][0]); acc[1][1] = fmaf(m1, sv.y, acc[1][1]);
            acc[1][2] = fmaf(m1, sv.z, acc[1][2]); acc[1][3] = fmaf(m1, sv.w, acc[1][3]);
        }
        __syncthreads();  // everyone is done reading S and M
        const float* st = ws_tilde + off;
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            const float4 t4 = *reinterpret_cast<const float4*>(st + (r + a) * kDim + c0 + cc);
            *reinterpret_cast<float4*>(S + (r + a) * kCombineCols + cc) =
                make_float4(acc[a][0] + t4.x, acc[a][1] + t4.y, acc[a][2] + t4.z, acc[a][3] + t4.w);
        }
        __syncthreads();
    }
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
                              float* final_state, const SegWorkspace& ws, int* status,
                              cudaStream_t stream, uint64_t* launches,
                              const int32_t* host_seqlens, float* ckpt, int ckpt_chunks,
                              const ProParams* pro) {
    if (num_seqs <= 0 || heads <= 0) return cudaSuccess;
    const int64_t units = (int64_t)num_seqs * heads;
    if (units > INT32_MAX) return cudaErrorInvalidValue;
    SeqOrder order;
    order.count = 0;
    order.num_seqs = num_seqs;
    order.total_tokens = total_tokens;
    order.total_slots = INT64_MAX;  // without host lengths only the token bound is checked
    order.total_ckpts = INT64_MAX;
    if (host_seqlens) {
        int64_t slots = 0, ckpts = 0;
        for (int n = 0; n < num_seqs; ++n) {
            const int ns = segment_plan(host_seqlens[n], heads).nseg;
            if (ns > 1) slots += ns;
            if (ckpt_chunks > 0) ckpts += host_seqlens[n] / (kChunk * ckpt_chunks);
        }
        order.total_slots = slots;
        order.total_ckpts = ckpts;
    }
    if (host_seqlens && num_seqs <= kMaxOrdered) {
        std::vector<int> idx(num_seqs);
        std::iota(idx.begin(), idx.end(), 0);
        auto nc = [&](int i) { return ((int64_t)host_seqlens[i] + kChunk - 1) / kChunk; };
        std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return nc(a) > nc(b); });
        for (int r = 0; r < num_seqs; ++r) {
            order.seq[r] = (uint16_t)idx[r];
            order.len[r] = host_seqlens[r];
        }
        order.count = num_seqs;
    }
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
    prm.ws_tilde = ws.tilde;
    prm.ws_trans = ws.trans;
    prm.ws_in = ws.in;
    prm.ckpt = ckpt_chunks > 0 ? ckpt : nullptr;
    prm.ckpt_chunks = ckpt_chunks > 0 ? ckpt_chunks : 1;
    prm.pro_A_log = pro ? pro->A_log : nullptr;
    prm.pro_dt_bias = pro ? pro->dt_bias : nullptr;
    prm.pro_lb = pro ? pro->lower_bound : 0.f;
    prm.pro_q_scale = pro ? pro->q_scale : 1.f;
    prm.H = heads;
    prm.pass = 0;
    if (pro && prm.ckpt) return cudaErrorInvalidValue;
    auto kernel = pro ? kda_prefill_tc_kernel<false, true>
                      : prm.ckpt ? kda_prefill_tc_kernel<true, false>
                                 : kda_prefill_tc_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const int zsplit = ws.max_segments > 1 ? 2 * (ws.max_segments - 1) : 1;
    // pass 0: whole sequences, and pass A (segment states and transitions) of split ones
    kernel<<<dim3((unsigned)units, 1, zsplit), kThreadsTC, SMEM_ALLOC, stream>>>(mq, mk, mv, mg,
                                                                                 prm, order);
    if (launches) ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess || ws.max_segments <= 1) return e;
    // compose the incoming state of every segment
    const int csmem = (kDim * kCombineLdM + kDim * kCombineCols) * 4;
    if ((e = cudaFuncSetAttribute(kda_segment_combine_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, csmem)) != cudaSuccess)
        return e;
    kda_segment_combine_kernel<<<dim3(num_seqs, heads, kCombineColBlocks), kCombineThreads, csmem,
                                 stream>>>(
        cu_seqlens, init_state, ws.tilde, ws.trans, ws.in, heads, status, order);
    if (launches) ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // pass B: every segment of the split sequences from its composed incoming state
    prm.pass = 1;
    kernel<<<dim3((unsigned)units, 1, ws.max_segments), kThreadsTC, SMEM_ALLOC, stream>>>(
        mq, mk, mv, mg, prm, order);
    if (launches) ++*launches;
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, cudaStream_t stream) {
    kda_wait_selftest_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace kda
