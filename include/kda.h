/*
 * kda.h — C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * The operation.  Each (sequence n, head h) unit keeps a d_k x d_v fp32 state S (rows are key
 * channels) and, token by token,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t,
 *
 * with alpha_t = exp(log_alpha_t) one retention factor per key channel and beta_t a scalar
 * write strength.  Source: "How Kimi K3 Engineered Its Way to the Frontier"
 * (codepointer.substack.com), section "How KDA updates its state" (the report's formula and
 * the three-line token loop of flash-linear-attention's naive.py); restated in "Kimi K3"
 * (ai.thesatyajit.com), section "Kimi Delta Attention: constant-size memory over a million
 * tokens".  The interface mirrors FlashKDA's forward as described there (section "FlashKDA:
 * the equation, shipped as a kernel"): q, k, v, gate, beta, optional state in and out,
 * variable-length batching through cumulative sequence lengths, d = 128.
 *
 * Conventions shared by every entry point
 *   - Layouts are row-major and contiguous, batch folded into tokens:
 *       q, k, log_alpha : [T_tot, H, d_k]     v, out : [T_tot, H, d_v]     beta : [T_tot, H]
 *       states          : fp32 [N, H, d_k, d_v], row = key channel
 *   - Element type of q, k, v, log_alpha, beta and out: bf16 (KDA_BF16) or fp32 (KDA_FP32).
 *     log_alpha is the natural-log gate (alpha = exp(log_alpha), expected <= 0); beta is the
 *     write strength itself (already passed through a sigmoid).  No scale is applied to q.
 *   - Only d_k = d_v = 128 is supported.
 *   - Device tensors that a kernel reads or writes as 16-byte vectors must be 16-byte aligned
 *     (every torch allocation is); each entry point states which, and a misaligned one returns
 *     KDA_ERR_INVALID_ARG.  The prefill entry points need it for q, k, v, log_alpha, out and
 *     the states.
 *   - Ownership: the caller owns and allocates every buffer (device memory unless marked
 *     host).  The library never allocates or frees memory and keeps no per-call state; its
 *     only globals are the sticky device status word read by kda_read_device_status(), the
 *     fixed scratch array behind kda_fwd_chunked_noalloc() and the three streams per device
 *     of kda_fwd_chunked_host().
 *   - Every compute entry point but kda_fwd_chunked_host is asynchronous on `stream` (NULL =
 *     legacy default stream).  Host-side argument checks are synchronous and return before
 *     anything is launched.
 *   - With KDA_NVTX=1 in the environment (read once per process), every compute entry point
 *     wraps its launches in an NVTX range named after the entry point.
 *   - Errors: KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED / KDA_ERR_WORKSPACE from the host
 *     checks, KDA_ERR_CUDA when a launch fails.  Conditions found on the device (a gate outside
 *     the supported domain, a bounded wait that gave up) set the sticky device status word;
 *     the kernels never trap or abort.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without CUDA headers. */
typedef struct CUstream_st* kda_stream_t;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, lengths not summing to T_tot     */
    KDA_ERR_UNSUPPORTED = -2,  /* d_k or d_v other than 128, unknown dtype                  */
    KDA_ERR_WORKSPACE = -3,    /* workspace missing or smaller than kda_fwd_workspace_bytes */
    KDA_ERR_CUDA = -4,         /* a CUDA launch or query failed                             */
    KDA_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up (device status word)   */
    KDA_ERR_DECAY_RANGE = -6   /* log_alpha > 0, or below -20 (see kda_fwd_chunked); in    */
                               /* kda_bwd, a 16-token chunk decaying beyond 160           */
} kda_status;

typedef enum kda_dtype { KDA_BF16 = 0, KDA_FP32 = 1 } kda_dtype;

/* Problem description.  host_seqlens is a HOST array of num_seqs lengths; it must equal the
 * differences of the device cu_seqlens array.  It lets the library size grids and workspace
 * without reading device memory.  The kernels check what they derive from the device array
 * against it before touching memory: a prefill CTA compares its sequence's length with the
 * host's (for calls of at most 2,048 sequences) and every derived offset (tokens, segment
 * workspace slots, checkpoint slots) with the host totals; the backward, decode-window and
 * fp32 prefill kernels check the token range and the workspace blocks.  A disagreement sets
 * KDA_ERR_INVALID_ARG in the device status word (read it with kda_read_device_status) and the
 * affected work item writes nothing. */
typedef struct kda_desc {
    int32_t num_seqs;            /* N >= 1                                            */
    int32_t num_heads;           /* H >= 1                                            */
    int64_t total_tokens;        /* T_tot = sum of host_seqlens                       */
    int32_t d_k;                 /* must be 128                                       */
    int32_t d_v;                 /* must be 128                                       */
    int32_t in_dtype;            /* kda_dtype of q, k, v, log_alpha, beta and out     */
    int32_t reserved;            /* must be 0                                         */
    const int32_t* host_seqlens; /* host, [num_seqs], each >= 0                       */
} kda_desc;

/* How a prefill call is split into work items (host-side plan, no device access). */
typedef struct kda_plan_info {
    int64_t chunks;           /* 64-token chunks summed over sequences (one head)          */
    int64_t work_items;       /* (sequence, segment) items per head                        */
    int32_t split_sequences;  /* sequences processed as more than one segment              */
    int32_t chunk_size;       /* tokens per chunk (64)                                     */
    int32_t segment_chunks;   /* longest segment of a split sequence, in chunks (0: none)  */
    int32_t reserved;
    size_t workspace_bytes;   /* what kda_fwd_chunked needs for this description           */
} kda_plan_info;

/*
 * kda_fwd_plan — fill *info with the work split of a prefill call.  Host only, no CUDA call.
 * Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_UNSUPPORTED.
 */
kda_status kda_fwd_plan(const kda_desc* desc, kda_plan_info* info);

/*
 * kda_fwd_workspace_bytes — bytes of device workspace kda_fwd_chunked needs for `desc`
 * (0 when no sequence is split into segments).  Host only.  Returns 0 for an invalid desc.
 */
size_t kda_fwd_workspace_bytes(const kda_desc* desc);

/*
 * kda_fwd_chunked — chunked prefill over packed variable-length sequences.
 *
 * Computes every o_t and, optionally, the final state of every (sequence, head) unit, exactly
 * as the token loop would, by the chunkwise form (64-token chunks aligned to each sequence's
 * own start; intra-chunk work as dense tensor-core tiles; one serial state step per chunk)
 * described in "How Kimi K3 Engineered Its Way to the Frontier", section "FlashKDA steps the
 * state once per 16 tokens".  Long sequences (above 65,536 tokens) are split into segments
 * whose transitions are evaluated independently of their incoming state and composed exactly
 * afterwards ("k3_training_and_infra_notes", section 4.1, intra-device context parallelism);
 * the segment count is a function of the sequence's length and the head count only (see
 * kda_fwd_plan), picked for the waves of GB300's 152 SMs.
 *
 *   desc          problem description (host)
 *   q, k, v, log_alpha, beta   device inputs, layouts above, element type desc->in_dtype
 *   init_state    device fp32 [N, H, 128, 128], or NULL for zeros.  May alias final_state.
 *   cu_seqlens    device int32 [N + 1], cu_seqlens[0] = 0, differences = host_seqlens
 *   out           device [T_tot, H, 128] of desc->in_dtype; must not alias any input
 *   final_state   device fp32 [N, H, 128, 128], or NULL to skip.  A zero-length sequence's
 *                 final state is its initial state.
 *   workspace     device scratch of at least kda_fwd_workspace_bytes(desc) bytes, 256-byte
 *                 aligned (NULL allowed when that size is 0).  Contents on entry are ignored.
 *   stream        CUDA stream the kernels are launched on.
 *
 * Bit-exactness: a sequence's results depend only on its own inputs and length, never on
 * the other sequences packed with it.
 *
 * Gate domain: every log_alpha in [-20, 0] is computed; this contains K3's bounded gate,
 * lower_bound * sigmoid(...) with lower_bound = -5 ("How Kimi K3 Engineered Its Way to the
 * Frontier", section "How KDA updates its state").  A chunk is a decay window: it starts where
 * the previous one ended, stays inside one 64-token block of the sequence, and is the longest
 * run of whole four-token groups (or the rest of the block) whose cumulative log-decay stays
 * within 80 in every channel, so every exponential factor of the chunkwise form is at most
 * e^40 in magnitude.  Ordinary gates give whole 64-token chunks; faster decay gives shorter
 * chunks (16 tokens at log_alpha = -5) and a proportionally slower call.  A positive log_alpha,
 * or a four-token group decaying by more than 80 in one channel (only possible below -20),
 * sets KDA_ERR_DECAY_RANGE in the device status word and leaves out and final_state
 * unspecified.  fp32 inputs (KDA_FP32) run the token loop itself in fp32, one pass over each
 * sequence, exact for every log_alpha <= 0 (no range applies).
 */
kda_status kda_fwd_chunked(const kda_desc* desc, const void* q, const void* k, const void* v,
                           const void* log_alpha, const void* beta, const float* init_state,
                           const int32_t* cu_seqlens, void* out, float* final_state,
                           void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_fwd_checkpoint_count — number of states kda_fwd_chunked_ckpt writes for `desc` and an
 * interval of `ckpt_every` tokens: the sum over sequences of floor(L_n / ckpt_every).  Host
 * only.  Returns -1 if the description is invalid or ckpt_every is not a positive multiple of
 * 64 (the chunk size).
 */
int64_t kda_fwd_checkpoint_count(const kda_desc* desc, int32_t ckpt_every);

/*
 * kda_fwd_chunked_ckpt — kda_fwd_chunked that also writes state checkpoints.
 *
 * A prefix cache can resume a sequence only where its recurrent state was saved, and serving
 * saves it at the block-aligned positions a prefix lookup can reference
 * ("k3_training_and_infra_notes", section 4.5, KDA-aware prefix cache management; "How Kimi K3
 * Engineered Its Way to the Frontier", section "KDA states and MLA KV blocks share one paged
 * pool", Figure 12: a checkpoint at a 512-token hash-block boundary).  For every (sequence,
 * head) this call writes the fp32 state after the first p tokens, for p = ckpt_every,
 * 2 ckpt_every, ... up to and including the sequence length, in the layout of final_state.
 *
 *   ckpt_every    positive multiple of 64 (the chunk size), in tokens
 *   ckpt_states   device fp32 [count, H, 128, 128], count = kda_fwd_checkpoint_count(desc,
 *                 ckpt_every): sequence by sequence, each sequence's positions in increasing
 *                 order.  Must not alias any other argument; NULL only when count is 0.
 * Everything else (arguments, layouts, errors) is as for kda_fwd_chunked, and the outputs and
 * final states are bit-identical to that call's.  bf16 inputs only (KDA_ERR_UNSUPPORTED for
 * fp32 inputs).
 */
kda_status kda_fwd_chunked_ckpt(const kda_desc* desc, const void* q, const void* k,
                                const void* v, const void* log_alpha, const void* beta,
                                const float* init_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, int32_t ckpt_every, float* ckpt_states,
                                void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_fwd_chunked_noalloc — kda_fwd_chunked for callers that cannot allocate device memory.
 *
 * No counterpart in the paper: this is a deployment convenience.  Some callers cannot supply
 * the scratch workspace kda_fwd_chunked asks for, because they may not call cudaMalloc where
 * they run (inside an allocator or memory-pool callback, in a host that forbids device
 * allocation, or on a latency-critical path where an allocation could synchronise the
 * device).  This variant takes the same arguments minus the workspace and uses a scratch array
 * built into the library instead; it allocates nothing and calls no allocating routine.
 *
 *   - The scratch array is KDA_NOALLOC_SCRATCH_BYTES (48 MiB) of device memory that every GPU
 *     which loads this library holds until the process exits.
 *   - A call whose kda_fwd_workspace_bytes(desc) exceeds KDA_NOALLOC_SCRATCH_BYTES returns
 *     KDA_ERR_WORKSPACE before launching anything (the workspace holds 3 x 64 KiB per head
 *     and segment, so with H = 16 heads 16 segments fit in total).  Calls that need no
 *     workspace always run.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; nothing in it has to
 *     start at zero.  Calls that overlap on the GPU (different streams, or different host
 *     threads) race on the array: serialise them.
 * Everything else — arguments, layouts, results, errors — is as for kda_fwd_chunked.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)
kda_status kda_fwd_chunked_noalloc(const kda_desc* desc, const void* q, const void* k,
                                   const void* v, const void* log_alpha, const void* beta,
                                   const float* init_state, const int32_t* cu_seqlens, void* out,
                                   float* final_state, kda_stream_t stream);

/*
 * kda_fwd_host_workspace_bytes — bytes of device workspace kda_fwd_chunked_host needs for
 * `desc` cut into `parts` token-range parts.  Host only.  Returns 0 for an invalid desc or
 * part count.
 *
 * kda_fwd_chunked_host — kda_fwd_chunked on HOST buffers: uploads the inputs, runs the prefill
 * and downloads the results, overlapping the three.
 *
 * No counterpart in the paper: a caller whose tensors live in host memory would otherwise copy
 * everything up, compute, and copy everything down in turn.  The host link is the bound of such
 * a call, so the tokens are cut into parts and three streams of the library's own (created per
 * device on first use, kept for the process) overlap the upload of one part, the kernels of the
 * previous part and the download of the part before that.  Part j covers tokens [b_j, b_{j+1})
 * of every sequence longer than b_j; the boundaries are multiples of the 64-token chunk chosen
 * so that the parts hold about equal token counts, and no part spans more than 65,536 tokens
 * of a sequence (so more parts than asked for can run).  Each part's kernels are one
 * kda_fwd_chunked call whose initial states are the previous part's final states: a sequence
 * cut by a boundary is computed as a prefill resumed from its saved fp32 state, which agrees
 * with one kda_fwd_chunked call within rounding, not bit for bit.  A sequence that lies inside
 * the first part (for example every sequence, with parts = 1) gets the bits of kda_fwd_chunked.
 *
 *   desc          problem description (host), as for kda_fwd_chunked
 *   q, k, v, log_alpha, beta   HOST inputs, layouts and element type as for kda_fwd_chunked.
 *                 Page-locked (pinned) memory lets the copies run asynchronously and overlap;
 *                 pageable memory gives the same results with the copies serialised.
 *   init_state    HOST fp32 [N, H, 128, 128], or NULL for zeros
 *   out           HOST [T_tot, H, 128] of desc->in_dtype; must not overlap an input
 *   final_state   HOST fp32 [N, H, 128, 128], or NULL to skip
 *   parts         token-range parts, 1..64, or 0 for 8
 *   workspace     device scratch of at least kda_fwd_host_workspace_bytes(desc, parts) bytes,
 *                 256-byte aligned: the states in flight, every part's cumulative lengths and
 *                 three slots of one part's inputs and outputs.  Contents on entry are ignored.
 *   stream        the call's work starts after the work already queued on this stream.
 * Unlike the device entry points the call is synchronous: it returns when out and final_state
 * hold the results (or, after an error, when every copy it issued has finished).  Errors are
 * those of kda_fwd_chunked, plus KDA_ERR_WORKSPACE for a missing or small workspace and
 * KDA_ERR_CUDA for a failed copy or stream call.
 */
size_t kda_fwd_host_workspace_bytes(const kda_desc* desc, int32_t parts);
kda_status kda_fwd_chunked_host(const kda_desc* desc, const void* q, const void* k,
                                const void* v, const void* log_alpha, const void* beta,
                                const float* init_state, void* out, float* final_state,
                                int32_t parts, void* workspace, size_t workspace_bytes,
                                kda_stream_t stream);

/*
 * kda_decode_step — one decode token per (sequence, head), state updated in place.
 *
 * For every unit: S <- Diag(exp(g)) S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q.
 * The state is read once and written once ("k3_training_and_infra_notes", section 4.5, KDA
 * decoding: the recurrent state is updated in place at every decoding step).
 *
 *   desc          num_seqs = N, total_tokens = N; host_seqlens may be NULL (all lengths 1)
 *   q, k, log_alpha  device [N, H, 128];  v: [N, H, 128];  beta: [N, H]  (desc->in_dtype)
 *   state         device fp32 [N, H, 128, 128], read and overwritten in place
 *   out           device [N, H, 128] of desc->in_dtype; must not alias any input
 */
kda_status kda_decode_step(const kda_desc* desc, const void* q, const void* k, const void* v,
                           const void* log_alpha, const void* beta, float* state, void* out,
                           kda_stream_t stream);

/*
 * kda_decode_window — a run of decode tokens per sequence in one pass over the state.
 *
 * Speculative decoding verifies a window of drafted tokens and must then move each state to
 * the last accepted token.  The state after any accepted prefix follows from the drafted
 * tokens' projected inputs, which are far smaller than the state, so only those are cached:
 * the accepted tokens are replayed on-chip together with the bonus token and the next draft
 * window in one recurrent loop, and the state is written back once
 * ("k3_training_and_infra_notes", section 4.5, KDA decoding).  For every (sequence, head):
 * starting from `state`, the tokens of sequence n (rows cu_seqlens[n] .. cu_seqlens[n+1] - 1)
 * run through the recurrence of kda_decode_step one after another; each token's output is
 * computed from the state after the tokens before it; the state after the first commit[n]
 * tokens is written back.
 *
 *   desc          num_seqs = N; host_seqlens required: per-sequence run lengths, 0 .. 64
 *   q, k, log_alpha, v  device [T, H, 128];  beta: [T, H]  (T = total_tokens, desc->in_dtype)
 *   cu_seqlens    device int32 [N + 1], differences = host_seqlens
 *   state         device fp32 [N, H, 128, 128]; overwritten with the state after the first
 *                 commit[n] tokens of run n, left untouched when that count is 0
 *   out           device [T, H, 128] of desc->in_dtype, or NULL to skip the outputs
 *   commit        device int32 [N] (each clamped to 0 .. run length), or NULL to commit every
 *                 token
 * A run of one token with commit 1 gives the bits of kda_decode_step.
 */
kda_status kda_decode_window(const kda_desc* desc, const void* q, const void* k, const void* v,
                             const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                             float* state, void* out, const int32_t* commit, kda_stream_t stream);

/*
 * Input prologue: the recurrence's inputs from a layer's raw per-token projections.
 *
 * Queries and keys of a KDA layer pass through Swish and are then L2-normalised over their
 * 128 channels; values pass through Swish ("Kimi K3" (ai.thesatyajit.com), section "Kimi Delta
 * Attention: constant-size memory over a million tokens").  The decay is K3's gate with a lower
 * bound, log_alpha = lower_bound * sigmoid(exp(A_log[h]) * (g_raw + dt_bias[h, :])), which keeps
 * every log_alpha inside (lower_bound, 0) ("How Kimi K3 Engineered Its Way to the Frontier",
 * section "How KDA updates its state").  beta arrives as logits and passes through a sigmoid
 * (FlashKDA's forward, section "FlashKDA: the equation, shipped as a kernel").  Readings where
 * the sources are silent: the L2 norm divides by sqrt(sum of squares + 1e-6); q is multiplied
 * by q_scale after its norm.  The short convolution that precedes Swish in the layer is the
 * caller's: the raw q, k, v here are its outputs.
 *
 * Arithmetic (fp32, every result rounded to bf16 where an unfused pipeline would store it):
 *   sigmoid(x) = 1 / (1 + 2^(-x log2 e)) with the hardware exp2 and reciprocal approximations
 *   (about 1e-6 relative error); Swish(x) = x sigmoid(x); the row norm sums the squares of eight
 *   consecutive channels in order and then adds the sixteen partial sums pairwise (strides 1,
 *   2, 4, 8).
 */
typedef struct {
  const float* A_log;    /* device fp32 [H]: per-head log decay rate */
  const float* dt_bias;  /* device fp32 [H, 128], or NULL for none */
  float lower_bound;     /* in [-80, 0): most negative log_alpha (K3 uses -5); the chunked
                            prefill computes log_alpha >= -20 (see kda_fwd_chunked) */
  float q_scale;         /* finite, > 0: factor on the normalised q (1/sqrt(128) is usual) */
} kda_prologue_params;

/*
 * kda_prologue — the prologue alone, as an elementwise pass over HBM (for decode steps and
 * windows, or any caller that wants the transformed inputs).
 *
 *   desc          total_tokens rows, num_heads heads; in_dtype must be KDA_BF16;
 *                 host_seqlens unused (may be NULL)
 *   q_raw, k_raw, v_raw, g_raw   device bf16 [T, H, 128]
 *   beta_logit    device bf16 [T, H]
 *   q, k, v, log_alpha           device bf16 [T, H, 128] outputs
 *   beta          device bf16 [T, H] output
 * Outputs must not alias inputs or each other.  Returns KDA_ERR_UNSUPPORTED for fp32 inputs.
 */
kda_status kda_prologue(const kda_desc* desc, const kda_prologue_params* prm, const void* q_raw,
                        const void* k_raw, const void* v_raw, const void* g_raw,
                        const void* beta_logit, void* q, void* k, void* v, void* log_alpha,
                        void* beta, kda_stream_t stream);

/*
 * kda_prologue_conv — the short convolution of q, k and v, then the prologue, as one pass.
 *
 * A KDA layer produces q, k and v by a short convolution followed by the prologue ("Kimi K3"
 * (ai.thesatyajit.com), section "Kimi Delta Attention…"); the convolution is causal and
 * depthwise with kernel size 4, and serving keeps three of its caches per request and layer
 * ("How Kimi K3 Engineered Its Way to the Frontier", section "What the hybrid saves": 216 KiB per
 * layer in bf16).  Per (sequence, head, channel): y_t = sum_{j=0..3} w[j] x_{t-3+j}, no bias,
 * w[3] on the current token, inputs before the sequence's first token from the cache (zeros when
 * cache_in is NULL); accumulated in fp32 in the order j = 0..3 and passed to the prologue
 * unrounded.  log_alpha and beta get no convolution.
 *
 *   desc          as for kda_fwd_chunked (host_seqlens required); in_dtype KDA_BF16
 *   conv->w_q, w_k, w_v   device fp32 [H, 128, 4], 16-byte aligned
 *   conv->cache_in        device bf16 [N, 3, 3, H, 128] (tensor q/k/v, then the 3 inputs before
 *                         each sequence, oldest first), or NULL for zeros
 *   conv->cache_out       device bf16, same layout: each sequence's last 3 raw inputs after the
 *                         call (continuing from cache_in when shorter), or NULL; may equal
 *                         cache_in (updated in place)
 *   cu_seqlens    device int32 [N+1]
 * Other arguments and outputs as for kda_prologue.  The outputs feed kda_fwd_chunked (or the
 * decode calls); a run split into consecutive calls with the cache carried equals one call.
 */
typedef struct {
  const float* w_q;      /* device fp32 [H, 128, 4] */
  const float* w_k;
  const float* w_v;
  const void* cache_in;  /* device bf16 [N, 3, 3, H, 128] or NULL */
  void* cache_out;       /* device bf16 [N, 3, 3, H, 128] or NULL; may equal cache_in */
} kda_conv_params;

kda_status kda_prologue_conv(const kda_desc* desc, const kda_prologue_params* prm,
                             const kda_conv_params* conv, const int32_t* cu_seqlens,
                             const void* q_raw, const void* k_raw, const void* v_raw,
                             const void* g_raw, const void* beta_logit, void* q, void* k, void* v,
                             void* log_alpha, void* beta, kda_stream_t stream);

/*
 * kda_fwd_chunked_prologue — kda_fwd_chunked on raw projections, with the prologue fused into
 * the prefill's load path: the transformed q, k, v, log_alpha and beta never go to HBM.
 *
 * Arguments as kda_fwd_chunked, with q_raw, k_raw, v_raw, g_raw and beta_logit (layouts as q, k,
 * v, log_alpha and beta) in place of the transformed inputs and `prm` as for kda_prologue.
 * Outputs and final states are bit-identical to kda_prologue followed by kda_fwd_chunked.
 * bf16 inputs only (KDA_ERR_UNSUPPORTED for fp32 inputs).
 */
kda_status kda_fwd_chunked_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                    const void* q_raw, const void* k_raw, const void* v_raw,
                                    const void* g_raw, const void* beta_logit,
                                    const float* init_state, const int32_t* cu_seqlens, void* out,
                                    float* final_state, void* workspace, size_t workspace_bytes,
                                    kda_stream_t stream);

/*
 * kda_decode_step_prologue, kda_decode_window_prologue — kda_decode_step and kda_decode_window
 * on raw projections, with the input prologue (as for kda_prologue) fused into the decode kernels:
 * K3's decode reads a token's projected inputs and normalises and gates them on-chip in the same
 * kernel as the recurrence ("k3_training_and_infra_notes", section 4.5, KDA decoding).
 *
 * Arguments as kda_decode_step / kda_decode_window, with q_raw, k_raw, v_raw, g_raw and
 * beta_logit in place of q, k, v, log_alpha and beta, and `prm` as for kda_prologue; q_raw and
 * k_raw must be 16-byte aligned (KDA_ERR_INVALID_ARG otherwise).  Outputs and states are
 * bit-identical to kda_prologue followed by the plain call.  bf16 inputs only
 * (KDA_ERR_UNSUPPORTED for fp32 inputs).
 */
kda_status kda_decode_step_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                    const void* q_raw, const void* k_raw, const void* v_raw,
                                    const void* g_raw, const void* beta_logit, float* state,
                                    void* out, kda_stream_t stream);
kda_status kda_decode_window_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                      const void* q_raw, const void* k_raw, const void* v_raw,
                                      const void* g_raw, const void* beta_logit,
                                      const int32_t* cu_seqlens, float* state, void* out,
                                      const int32_t* commit, kda_stream_t stream);

/*
 * kda_bwd — gradients of the recurrence (the backward pass) for training.
 *
 * For the forward of kda_fwd_chunked (the token loop of "How Kimi K3 Engineered Its Way to the
 * Frontier", section "How KDA updates its state") and the gradient d_out of a loss with respect to
 * every output (and optionally d_state with respect to the final states), returns the gradients
 * with respect to q, k, v, log_alpha, beta and the initial states.  Chunked by 16 tokens (the
 * pages' state step, "FlashKDA steps the state once per 16 tokens"), on tensor cores (tf32
 * operands, fp32 accumulation): a forward pass stores the state at every chunk start, a reverse
 * pass carries the gradient of the state backwards and computes each chunk's gradients.
 * Domain: in every 16-token chunk, every key channel decays by at most 160 (a mean log_alpha of
 * -10 per token, twice the bounded gate's floor of -5); a chunk beyond that sets
 * KDA_ERR_DECAY_RANGE in the device status word and its gradients are then unspecified.
 *
 *   desc          as for kda_fwd_chunked (host_seqlens required); q, k, v, log_alpha, beta of
 *                 desc->in_dtype, layouts as there; q, k, v, log_alpha 16-byte aligned
 *   init_state    device fp32 [N, H, 128, 128] or NULL (zeros)
 *   d_out         device fp32 [T, H, 128]
 *   d_state       device fp32 [N, H, 128, 128] or NULL (no loss on the final states)
 *   dq, dk, dv, dlog_alpha   device fp32 [T, H, 128]; dbeta device fp32 [T, H];
 *   dinit_state   device fp32 [N, H, 128, 128]
 *   workspace     device, at least kda_bwd_workspace_bytes(desc) bytes, 16-byte aligned: the
 *                 sequences' chunk offsets, then per 16-token chunk and head three 16 x 16 fp32
 *                 tiles, the chunk's start state (128 x 128 fp32) and a 16 x 128 fp32 tile;
 *                 contents on return are unspecified
 * The gradients are deterministic (no atomics; every sum runs in a fixed order).  If the device
 * cu_seqlens disagree with the host lengths in their chunk total or run past T, the first launch
 * sets KDA_ERR_INVALID_ARG in the device status word, nothing else is computed and every output
 * is unspecified.  Outputs must not alias inputs or each other.  Argument, alignment and
 * workspace errors return KDA_ERR_INVALID_ARG / KDA_ERR_WORKSPACE before anything is launched.
 */
size_t kda_bwd_workspace_bytes(const kda_desc* desc);
kda_status kda_bwd(const kda_desc* desc, const void* q, const void* k, const void* v,
                   const void* log_alpha, const void* beta, const float* init_state,
                   const int32_t* cu_seqlens, const float* d_out, const float* d_state, float* dq,
                   float* dk, float* dv, float* dlog_alpha, float* dbeta, float* dinit_state,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_selftest_wait_timeout — diagnostic: launch one CTA that waits, through the kernels' own
 * bounded-wait code, on a barrier phase nothing completes.  The wait gives up after its limit
 * (about 2 s) and records KDA_ERR_TIMEOUT in the sticky status word, which
 * kda_read_device_status() then returns; the context stays usable.  Every wait of the compute
 * kernels is bounded the same way, so a lost arrival (a defect, or a fault elsewhere) ends as a
 * status code rather than a hang.  Returns KDA_OK once launched.
 */
kda_status kda_selftest_wait_timeout(kda_stream_t stream);

/*
 * kda_read_device_status — synchronise `stream`, then return and clear the sticky device
 * status word of the current device (KDA_OK when no kernel reported a problem).
 */
kda_status kda_read_device_status(kda_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* kda_status_string(kda_status status);

/* Number of kernels this library has launched in this process (all devices, all streams). */
uint64_t kda_launch_count(void);

/* Library ABI version (increments on any signature change). */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
