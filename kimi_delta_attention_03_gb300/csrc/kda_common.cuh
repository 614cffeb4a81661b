// kda_common.cuh — small device helpers shared by the KDA kernels of this library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kDim = 128;     // d_k = d_v
constexpr int kChunk = 64;    // tokens per chunk of the prefill path

// Segment plan of the prefill (intra-device context parallelism).  A sequence longer than
// kSplitChunks chunks is cut into segments: a first launch computes every segment's state from
// zero and its transition (two work items per segment but the last), a second reruns every
// segment from its composed incoming state (one item each).  A split sequence therefore costs
// about three passes over its tokens, so only sequences whose single pass would outlast a
// typical batch (above 64K tokens) are split.  The segment count is picked among a few
// candidates (128-chunk segments, and one, two or three items per SM per head) by a model of
// the two launches' waves on kPlanSMs SMs, segments of at least kMinSegChunks chunks: a wave of
// items costs its segment length, outputs 43 and no outputs 40 per chunk.  The plan is a
// function of the sequence's own length and the head count only, so packing never changes a
// sequence's results.  All segments but the last have seg_chunks chunks; the last is shorter
// or equal and never empty.
constexpr int kSplitChunks = 1024;
constexpr int kPlanSMs = 152;
constexpr int kMinSegChunks = 64;
struct SegPlan {
    int nseg;        // 1: the sequence runs whole
    int seg_chunks;  // chunks per segment (the last may have fewer)
};
__host__ __device__ __forceinline__ int64_t segment_plan_cost(int64_t nc, int H, int64_t n) {
    const int64_t seg = (nc + n - 1) / n;
    const int64_t w0 = (2 * (int64_t)H * (n - 1) + kPlanSMs - 1) / kPlanSMs;
    const int64_t w1 = ((int64_t)H * n + kPlanSMs - 1) / kPlanSMs;
    return seg * (40 * w0 + 43 * w1);
}
__host__ __device__ __forceinline__ SegPlan segment_plan(int64_t len, int H) {
    const int64_t nc = (len + kChunk - 1) / kChunk;
    if (nc <= kSplitChunks) return SegPlan{1, (int)nc};
    const int64_t cap = nc / kMinSegChunks;
    int64_t pick = (nc + 127) / 128;
    int64_t best = segment_plan_cost(nc, H, pick);
    for (int k = 1; k <= 3; ++k) {
        int64_t n = (int64_t)k * kPlanSMs / (H > 0 ? H : 1);
        n = n < cap ? n : cap;
        n = n > 2 ? n : 2;
        const int64_t c = segment_plan_cost(nc, H, n);
        if (c < best) {
            best = c;
            pick = n;
        }
    }
    const int64_t seg = (nc + pick - 1) / pick;
    return SegPlan{(int)((nc + seg - 1) / seg), (int)seg};
}

// Device status codes written into the sticky status word (same values as kda_status).
constexpr int kStatusDecayRange = KDA_ERR_DECAY_RANGE;
constexpr int kStatusTimeout = KDA_ERR_TIMEOUT;

// Record a device-side condition; the first one written stays until the host clears it.
__device__ __forceinline__ void report_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

template <typename T> struct io;

template <> struct io<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

template <> struct io<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// Two fp32 products (or fused multiply-adds) in one packed instruction, each rounded as its
// scalar form is: the same bits, half the issue slots.
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace kda

// Launchers implemented in the kernel translation units (called by kda_api.cu).
namespace kda {

// Workspace of the segmented prefill: three arrays of [slots][H][128][128] fp32 (segment
// states from zero, segment transitions, composed incoming states).
struct SegWorkspace {
    float* tilde;
    float* trans;
    float* in;
    int max_segments;  // 1 when no sequence is split (the workspace is then unused)
};

// The host's plan of a prefill call, passed by value to its kernels.
//  - Dispatch order of the CTAs: sequences ranked by chunk count, longest first (ties in packing
//    order), so that the longest units start in the first wave.  Only the order in which units
//    are scheduled changes; every unit computes the same bits wherever it runs.
//  - The host's sequence lengths and totals, against which every CTA checks what it derives from
//    the device cu_seqlens before it touches memory (a disagreement sets KDA_ERR_INVALID_ARG and
//    the CTA returns): its own length (when the call has at most kMaxOrdered sequences), and the
//    bounds of every derived offset (tokens, segment workspace slots, checkpoint slots).
constexpr int kMaxOrdered = 2048;
struct SeqOrder {
    int32_t count;                  // ranked sequences; 0 = packing order, no lengths below
    int32_t num_seqs;
    int64_t total_tokens;           // host T_tot
    int64_t total_slots;            // host segment workspace slots (per head)
    int64_t total_ckpts;            // host checkpoint count (per head), when checkpoints are written
    uint16_t seq[kMaxOrdered];      // seq[rank] = sequence index
    int32_t len[kMaxOrdered];       // len[n] = host length of sequence n (when count > 0)
};

// Input prologue parameters (raw projections in; see kda_prologue.cuh).
struct ProParams {
    const float* A_log;    // [H]
    const float* dt_bias;  // [H][128] or null
    float lower_bound;
    float q_scale;
};

// host_seqlens (optional, host memory): the sequence lengths, used only to rank the sequences
// for dispatch; without them the CTAs run in packing order.  ckpt (optional, device): state
// checkpoints after every ckpt_chunks chunks of each sequence, [count][H][128][128] fp32.
// pro (optional): q, k, v, g and beta are raw projections and the prologue runs in the kernel
// (not combined with checkpoints).
cudaError_t launch_prefill_tc(int num_seqs, int heads, int64_t total_tokens, const void* q,
                              const void* k, const void* v, const void* g, const void* beta,
                              const float* init_state, const int32_t* cu_seqlens, void* out,
                              float* final_state, const SegWorkspace& ws, int* status,
                              cudaStream_t stream, uint64_t* launches,
                              const int32_t* host_seqlens = nullptr, float* ckpt = nullptr,
                              int ckpt_chunks = 0, const ProParams* pro = nullptr);

// Decode step and window; pro (optional, bf16 only): the inputs are raw projections and the
// prologue runs in the kernel.
cudaError_t launch_decode(int dtype, int64_t units, int heads, const void* q, const void* k,
                          const void* v, const void* g, const void* beta, float* state,
                          void* out, int* status, cudaStream_t stream,
                          const ProParams* pro = nullptr);

// The state is read from state_in (zeros when null) and written to state_out (skipped when
// null); they may be the same array.  Also the prefill of fp32 inputs (commit null).  A unit
// whose device cu_seqlens run leaves [0, total_tokens) or exceeds max_len tokens sets
// KDA_ERR_INVALID_ARG in *status and is skipped.
cudaError_t launch_decode_window(int dtype, int num_seqs, int heads, const void* q,
                                 const void* k, const void* v, const void* g, const void* beta,
                                 const int32_t* cu_seqlens, const float* state_in,
                                 float* state_out, void* out, const int32_t* commit,
                                 int64_t total_tokens, int max_len, int* status,
                                 cudaStream_t stream, const ProParams* pro = nullptr);

// The prologue alone over `rows` (token, head) rows, bf16 in and out.
cudaError_t launch_prologue(int64_t rows, int heads, const void* q_raw, const void* k_raw,
                            const void* v_raw, const void* g_raw, const void* beta_logit,
                            const float* A_log, const float* dt_bias, float lower_bound,
                            float q_scale, void* q, void* k, void* v, void* g, void* beta,
                            cudaStream_t stream);

// Gradients of the recurrence, chunked by 16 tokens.  `chunks` is the host's chunk total (sum over
// the sequences of ceil(len / 16)); work holds backward_workspace_floats(num_seqs, heads, chunks)
// floats: the chunk offsets of the sequences and a stop flag, then per (chunk, head) the 16 x 16
// tiles T, P and At, then per (chunk, head) the state at the chunk's start and R = V - K_f S.
size_t backward_workspace_floats(int num_seqs, int heads, int64_t chunks);
int64_t backward_chunks(const int32_t* host_seqlens, int num_seqs);
cudaError_t launch_backward(int dtype, int num_seqs, int heads, const void* q, const void* k,
                            const void* v, const void* g, const void* beta,
                            const int32_t* cu_seqlens, const float* init_state,
                            const float* d_out, const float* d_state, float* dq, float* dk,
                            float* dv, float* dg, float* dbeta, float* d_init, float* work,
                            int64_t chunks, int64_t total_tokens, int* status,
                            cudaStream_t stream);

// One CTA whose bounded wait runs out: the status word then reads KDA_ERR_TIMEOUT.
cudaError_t launch_wait_selftest(int* status, cudaStream_t stream);

// The short convolution (kernel 4, cached) and the prologue over `rows` (token, head) rows; the
// cache after the call is written when cache_out is given (it may equal cache_in).
cudaError_t launch_prologue_conv(int64_t rows, int heads, int num_seqs, const void* q_raw,
                                 const void* k_raw, const void* v_raw, const void* g_raw,
                                 const void* beta_logit, const float* A_log, const float* dt_bias,
                                 float lower_bound, float q_scale, const float* w_q,
                                 const float* w_k, const float* w_v, const void* cache_in,
                                 void* cache_out, const int32_t* cu_seqlens, void* q, void* k,
                                 void* v, void* g, void* beta, cudaStream_t stream);
}  // namespace kda
