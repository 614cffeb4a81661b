/*
 * kda_oracle.c — fp64 CPU oracle for the Kimi Delta Attention (KDA) forward recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct definition that the
 * CUDA library is checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It includes no header of the CUDA library and shares no code,
 * table or constant with it; the product path never calls it.
 *
 * What it computes (per sequence n, per head h, tokens in sequence order):
 *
 *   S  <- Diag(exp(g_t)) S                 forget: key-channel rows decay
 *   u  <- v_t - S^T k_t                    the gap between what S returns for k_t and v_t
 *   S  <- S + (beta_t k_t) u^T             erase-and-write (delta rule)
 *   o_t <- S^T q_t                         read
 *
 * This is the three-line token loop of flash-linear-attention's fla/ops/kda/naive.py as shown
 * on "How Kimi K3 Engineered Its Way to the Frontier" (section "How KDA updates its state"),
 * and it equals the report's closed form
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t
 * (same page, same section; restated in "Kimi K3" on ai.thesatyajit.com, section
 * "Kimi Delta Attention: constant-size memory over a million tokens"), with g_t = log alpha_t.
 * Shapes follow the same section: S is [N, H, d_k, d_v] with a row per key channel, and the
 * gate g has one value per key channel per token per head.
 *
 * Precision: every input is widened exactly to double; nothing is rounded on the way out.
 * Parallelism: OpenMP over independent (sequence, head) units only; the per-unit arithmetic
 * order is the plain loop order, so results are bitwise reproducible run to run.
 *
 * Pins (tests/test_oracle_pins.py): exact rational brute force of the product of transition
 * matrices (T <= 8, d = 4); beta = 0 freezing; linear-attention reduction with orthonormal
 * keys; scalar gate == single-gate delta rule (and per-channel gate != swapped order);
 * delta-rule retrieval; segment composition; fixed state size.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Input element formats accepted by the oracle. */
enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 };

/* Exact widening of one stored element to double.  bf16 is the upper half of an IEEE
 * binary32, so shifting its 16 bits up gives the float it denotes. */
static double widen(const void* base, int fmt, int64_t idx) {
    if (fmt == ORACLE_F64) return ((const double*)base)[idx];
    if (fmt == ORACLE_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Row of the compact output array that receives token t, or -1 when t is not recorded.
 * With no windows every token is recorded at row t. */
static int64_t output_row(int64_t t, int32_t n_windows, const int64_t* windows) {
    if (n_windows == 0) return t;
    int64_t base = 0;
    for (int32_t w = 0; w < n_windows; ++w) {
        int64_t lo = windows[2 * w], hi = windows[2 * w + 1];
        if (t >= lo && t < hi) return base + (t - lo);
        base += hi - lo;
    }
    return -1;
}

/*
 * kda_oracle_recurrence
 *
 *   total_tokens  T_tot = cu_seqlens[num_seqs]
 *   cu_seqlens    [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0
 *   in_format     ORACLE_F64 / ORACLE_F32 / ORACLE_BF16 for q, k, v, g, beta
 *   q, k, g       [T_tot, num_heads, dk]   (g = natural-log decay, alpha = exp(g))
 *   v             [T_tot, num_heads, dv]
 *   beta          [T_tot, num_heads]       (write strength, already in (0,1))
 *   state_in      [num_seqs, num_heads, dk, dv] doubles, or NULL for zeros
 *   out           [rows, num_heads, dv] doubles, or NULL; rows = T_tot when n_windows = 0,
 *                 else the tokens of the windows [lo, hi) (global token indices) in order
 *   state_out     [num_seqs, num_heads, dk, dv] doubles, or NULL
 *   num_threads   OpenMP threads (<= 0: runtime default)
 *
 * Returns 0 on success, -1 on an invalid argument.
 */
int kda_oracle_recurrence(int64_t total_tokens, int32_t num_seqs, int32_t num_heads,
                          int32_t dk, int32_t dv, const int32_t* cu_seqlens, int32_t in_format,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const double* state_in, double* out,
                          int32_t n_windows, const int64_t* windows, double* state_out,
                          int32_t num_threads) {
    if (num_seqs < 0 || num_heads <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    if (in_format < ORACLE_F64 || in_format > ORACLE_BF16) return -1;
    if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[num_seqs] != total_tokens) return -1;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta)) return -1;
    if (n_windows < 0 || (n_windows > 0 && !windows)) return -1;

    const int64_t units = (int64_t)num_seqs * num_heads;
    const int64_t sdim = (int64_t)dk * dv;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t n = (int32_t)(unit / num_heads);
        const int32_t h = (int32_t)(unit % num_heads);
        double* S = (double*)malloc(sizeof(double) * sdim);
        double* u = (double*)malloc(sizeof(double) * dv);
        double* kt = (double*)malloc(sizeof(double) * dk);
        if (!S || !u || !kt) {
            free(S); free(u); free(kt);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        if (state_in)
            memcpy(S, state_in + unit * sdim, sizeof(double) * sdim);
        else
            memset(S, 0, sizeof(double) * sdim);

        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const int64_t kbase = (t * num_heads + h) * (int64_t)dk;
            const int64_t vbase = (t * num_heads + h) * (int64_t)dv;
            const double b = widen(beta, in_format, t * num_heads + h);

            /* forget: S <- Diag(exp(g_t)) S, one retention factor per key channel (row) */
            for (int32_t i = 0; i < dk; ++i) {
                const double a = exp(widen(g, in_format, kbase + i));
                for (int32_t j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= a;
            }
            /* erase target: u = v_t - S^T k_t */
            for (int32_t i = 0; i < dk; ++i) kt[i] = widen(k, in_format, kbase + i);
            for (int32_t j = 0; j < dv; ++j) u[j] = 0.0;
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) u[j] += kt[i] * S[(int64_t)i * dv + j];
            for (int32_t j = 0; j < dv; ++j) u[j] = widen(v, in_format, vbase + j) - u[j];
            /* write: S <- S + (beta_t k_t) u^T */
            for (int32_t i = 0; i < dk; ++i) {
                const double bk = b * kt[i];
                for (int32_t j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += bk * u[j];
            }
            /* read: o_t = S^T q_t */
            if (out) {
                const int64_t row = output_row(t, n_windows, windows);
                if (row >= 0) {
                    double* o = out + (row * num_heads + h) * (int64_t)dv;
                    for (int32_t j = 0; j < dv; ++j) o[j] = 0.0;
                    for (int32_t i = 0; i < dk; ++i) {
                        const double qi = widen(q, in_format, kbase + i);
                        for (int32_t j = 0; j < dv; ++j) o[j] += qi * S[(int64_t)i * dv + j];
                    }
                }
            }
        }
        if (state_out) memcpy(state_out + unit * sdim, S, sizeof(double) * sdim);
        free(S); free(u); free(kt);
    }
    return failed ? -1 : 0;
}

/* Version tag so a stale build is easy to spot. */
int kda_oracle_version(void) { return 1; }
