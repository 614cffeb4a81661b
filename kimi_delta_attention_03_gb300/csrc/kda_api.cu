// kda_api.cu — the C ABI declared in include/kda.h: host-side checks, the work plan, the
// sticky device status word, and the kernel launches.  No allocation happens here.
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "kda_common.cuh"

namespace {

std::atomic<uint64_t> g_launches{0};

// Optional NVTX ranges, one per entry-point call, named after the entry point, so that a
// profiler's timeline shows which library call launched which kernels.  Enabled by KDA_NVTX=1 in
// the environment (read once per process); otherwise a call costs one branch.
bool nvtx_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("KDA_NVTX");
        return e && e[0] == '1';
    }();
    return on;
}
struct NvtxRange {
    bool on;
    explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxRange() {
        if (on) nvtxRangePop();
    }
};

// One sticky status word per device; kernels write it with atomicCAS(0 -> code).
__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

// Vector loads and stores need 16-byte aligned tensors (torch allocations are 256-aligned).
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_desc(const kda_desc* d, bool need_lengths) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->d_k != 128 || d->d_v != 128) return KDA_ERR_UNSUPPORTED;
    if (d->in_dtype != KDA_BF16 && d->in_dtype != KDA_FP32) return KDA_ERR_UNSUPPORTED;
    if (d->num_seqs < 1 || d->num_heads < 1 || d->total_tokens < 0 || d->reserved != 0)
        return KDA_ERR_INVALID_ARG;
    if (need_lengths) {
        if (!d->host_seqlens) return KDA_ERR_INVALID_ARG;
        int64_t sum = 0;
        for (int32_t n = 0; n < d->num_seqs; ++n) {
            if (d->host_seqlens[n] < 0) return KDA_ERR_INVALID_ARG;
            sum += d->host_seqlens[n];
        }
        if (sum != d->total_tokens) return KDA_ERR_INVALID_ARG;
        // token offsets are formed as int32 cu_seqlens
        if (d->total_tokens > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    }
    return KDA_OK;
}

// The prologue's parameters: a per-head rate, an optional 16-byte aligned bias, a finite lower
// bound in [-80, 0) (so one token's decay stays inside the prefill's exponent range) and a
// finite positive q scale.
bool check_prologue(const kda_prologue_params* prm) {
    if (!prm || !prm->A_log || !aligned16(prm->dt_bias)) return false;
    if (!std::isfinite(prm->lower_bound) || prm->lower_bound >= 0.f || prm->lower_bound < -80.f)
        return false;
    return std::isfinite(prm->q_scale) && prm->q_scale > 0.f;
}

kda_status decode_step_impl(const kda_desc* desc, const void* q, const void* k,
                                   const void* v, const void* log_alpha, const void* beta,
                                   float* state, void* out, kda_stream_t stream,
                                   const kda_prologue_params* pro) {
    kda_status st = check_desc(desc, false);
    if (st != KDA_OK) return st;
    kda::ProParams pp = {};
    if (pro) {
        if (desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
        if (!check_prologue(pro)) return KDA_ERR_INVALID_ARG;
        pp = {pro->A_log, pro->dt_bias, pro->lower_bound, pro->q_scale};
    }
    // the fused prologue reads q and k rows as 16-byte vectors
    if (pro && (!aligned16(q) || !aligned16(k))) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens != desc->num_seqs) return KDA_ERR_INVALID_ARG;
    if (desc->host_seqlens) {
        for (int32_t n = 0; n < desc->num_seqs; ++n)
            if (desc->host_seqlens[n] != 1) return KDA_ERR_INVALID_ARG;
    }
    if (!q || !k || !v || !log_alpha || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    if (out == q || out == k || out == v || out == log_alpha || out == beta ||
        out == (const void*)state)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state)) return KDA_ERR_INVALID_ARG;
    int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    const int64_t units = (int64_t)desc->num_seqs * desc->num_heads;
    cudaError_t e = kda::launch_decode(desc->in_dtype, units, desc->num_heads, q, k, v,
                                       log_alpha, beta, state, out, status,
                                       (cudaStream_t)stream, pro ? &pp : nullptr);
    g_launches += 1;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status decode_window_impl(const kda_desc* desc, const void* q, const void* k,
                                     const void* v, const void* log_alpha, const void* beta,
                                     const int32_t* cu_seqlens, float* state, void* out,
                                     const int32_t* commit, kda_stream_t stream,
                                     const kda_prologue_params* pro) {
    kda_status st = check_desc(desc, true);
    if (st != KDA_OK) return st;
    kda::ProParams pp = {};
    if (pro) {
        if (desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
        if (!check_prologue(pro)) return KDA_ERR_INVALID_ARG;
        pp = {pro->A_log, pro->dt_bias, pro->lower_bound, pro->q_scale};
    }
    for (int32_t n = 0; n < desc->num_seqs; ++n)
        if (desc->host_seqlens[n] > 64) return KDA_ERR_INVALID_ARG;
    // the fused prologue reads q and k rows as 16-byte vectors
    if (pro && (!aligned16(q) || !aligned16(k))) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !state) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta)) return KDA_ERR_INVALID_ARG;
    if (out && (out == q || out == k || out == v || out == log_alpha || out == beta ||
                out == (const void*)state))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state)) return KDA_ERR_INVALID_ARG;
    int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    cudaError_t e = kda::launch_decode_window(desc->in_dtype, desc->num_seqs, desc->num_heads, q, k,
                                              v, log_alpha, beta, cu_seqlens, state, state, out,
                                              commit, desc->total_tokens, 64, status,
                                              (cudaStream_t)stream, pro ? &pp : nullptr);
    g_launches += 1;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status kda_fwd_plan(const kda_desc* desc, kda_plan_info* info) {
    if (!info) return KDA_ERR_INVALID_ARG;
    kda_status st = check_desc(desc, true);
    if (st != KDA_OK) return st;
    kda_plan_info p = {};
    p.chunk_size = kda::kChunk;
    p.segment_chunks = 0;
    int64_t slots = 0;
    for (int32_t n = 0; n < desc->num_seqs; ++n) {
        const int64_t L = desc->host_seqlens[n];
        const kda::SegPlan sp = kda::segment_plan(L, desc->num_heads);
        p.chunks += (L + kda::kChunk - 1) / kda::kChunk;
        p.work_items += sp.nseg;
        if (sp.nseg > 1) {
            p.split_sequences += 1;
            slots += sp.nseg;
            p.segment_chunks = std::max(p.segment_chunks, sp.seg_chunks);
        }
    }
    // three fp32 arrays [slots][H][128][128], each 256-byte aligned
    const size_t per = (size_t)slots * desc->num_heads * 128 * 128 * sizeof(float);
    p.workspace_bytes = slots ? 3 * per : 0;
    *info = p;
    return KDA_OK;
}

size_t kda_fwd_workspace_bytes(const kda_desc* desc) {
    kda_plan_info p;
    if (kda_fwd_plan(desc, &p) != KDA_OK) return 0;
    return p.workspace_bytes;
}

}  // extern "C"

namespace {

// kda_fwd_chunked with optional state checkpoints every ckpt_every tokens (0: none).
kda_status fwd_chunked_impl(const kda_desc* desc, const void* q, const void* k, const void* v,
                            const void* log_alpha, const void* beta, const float* init_state,
                            const int32_t* cu_seqlens, void* out, float* final_state,
                            int32_t ckpt_every, float* ckpt_states, void* workspace,
                            size_t workspace_bytes, kda_stream_t stream,
                            const kda_prologue_params* pro = nullptr) {
    kda_plan_info plan;
    kda_status st = kda_fwd_plan(desc, &plan);
    if (st != KDA_OK) return st;
    kda::ProParams pp = {};
    if (pro) {
        if (desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
        if (!check_prologue(pro)) return KDA_ERR_INVALID_ARG;
        pp = {pro->A_log, pro->dt_bias, pro->lower_bound, pro->q_scale};
    }
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !out))
        return KDA_ERR_INVALID_ARG;
    if (out && (out == q || out == k || out == v || out == log_alpha || out == beta))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
        !aligned16(out) || !aligned16(init_state) || !aligned16(final_state))
        return KDA_ERR_INVALID_ARG;
    int64_t ckpts = 0;
    if (ckpt_every != 0) {
        ckpts = kda_fwd_checkpoint_count(desc, ckpt_every);
        if (ckpts < 0) return KDA_ERR_INVALID_ARG;
        if (ckpts > 0 && desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
        if (ckpts > 0 && (!ckpt_states || !aligned16(ckpt_states))) return KDA_ERR_INVALID_ARG;
        const void* c = ckpt_states;
        if (ckpts > 0 && (c == q || c == k || c == v || c == log_alpha || c == beta || c == out ||
                          c == init_state || c == final_state))
            return KDA_ERR_INVALID_ARG;
    }
    if (plan.workspace_bytes > 0 && (!workspace || workspace_bytes < plan.workspace_bytes ||
                                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return KDA_ERR_WORKSPACE;
    int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    uint64_t launches = 0;
    cudaError_t e;
    kda::SegWorkspace ws = {nullptr, nullptr, nullptr, 1};
    if (plan.workspace_bytes > 0) {
        const size_t per = plan.workspace_bytes / 3;
        ws.tilde = static_cast<float*>(workspace);
        ws.trans = reinterpret_cast<float*>(static_cast<char*>(workspace) + per);
        ws.in = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * per);
        for (int32_t n = 0; n < desc->num_seqs; ++n)
            ws.max_segments = std::max(ws.max_segments,
                                       kda::segment_plan(desc->host_seqlens[n], desc->num_heads).nseg);
    }
    if (desc->in_dtype == KDA_BF16)
        e = kda::launch_prefill_tc(desc->num_seqs, desc->num_heads, desc->total_tokens, q, k, v,
                                   log_alpha, beta, init_state, cu_seqlens, out, final_state, ws,
                                   status, (cudaStream_t)stream, &launches,
                                   desc->host_seqlens, ckpts > 0 ? ckpt_states : nullptr,
                                   ckpts > 0 ? ckpt_every / kda::kChunk : 0, pro ? &pp : nullptr);
    else {  // fp32 inputs: the token loop in fp32 over whole sequences (exact for every gate)
        e = kda::launch_decode_window(desc->in_dtype, desc->num_seqs, desc->num_heads, q, k, v,
                                      log_alpha, beta, cu_seqlens, init_state, final_state, out,
                                      nullptr, desc->total_tokens, INT32_MAX, status,
                                      (cudaStream_t)stream);
        ++launches;
    }
    g_launches += launches;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status kda_fwd_chunked(const kda_desc* desc, const void* q, const void* k, const void* v,
                           const void* log_alpha, const void* beta, const float* init_state,
                           const int32_t* cu_seqlens, void* out, float* final_state,
                           void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_fwd_chunked");
    return fwd_chunked_impl(desc, q, k, v, log_alpha, beta, init_state, cu_seqlens, out,
                            final_state, 0, nullptr, workspace, workspace_bytes, stream);
}

int64_t kda_fwd_checkpoint_count(const kda_desc* desc, int32_t ckpt_every) {
    if (ckpt_every <= 0 || ckpt_every % kda::kChunk != 0) return -1;
    if (check_desc(desc, true) != KDA_OK) return -1;
    int64_t count = 0;
    for (int32_t n = 0; n < desc->num_seqs; ++n) count += desc->host_seqlens[n] / ckpt_every;
    return count;
}

kda_status kda_fwd_chunked_ckpt(const kda_desc* desc, const void* q, const void* k,
                                const void* v, const void* log_alpha, const void* beta,
                                const float* init_state, const int32_t* cu_seqlens, void* out,
                                float* final_state, int32_t ckpt_every, float* ckpt_states,
                                void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_fwd_chunked_ckpt");
    if (ckpt_every <= 0) return KDA_ERR_INVALID_ARG;
    return fwd_chunked_impl(desc, q, k, v, log_alpha, beta, init_state, cu_seqlens, out,
                            final_state, ckpt_every, ckpt_states, workspace, workspace_bytes,
                            stream);
}

kda_status kda_fwd_chunked_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                    const void* q_raw, const void* k_raw, const void* v_raw,
                                    const void* g_raw, const void* beta_logit,
                                    const float* init_state, const int32_t* cu_seqlens, void* out,
                                    float* final_state, void* workspace, size_t workspace_bytes,
                                    kda_stream_t stream) {
    NvtxRange nvtx_range("kda_fwd_chunked_prologue");
    if (!prm) return KDA_ERR_INVALID_ARG;
    return fwd_chunked_impl(desc, q_raw, k_raw, v_raw, g_raw, beta_logit, init_state, cu_seqlens,
                            out, final_state, 0, nullptr, workspace, workspace_bytes, stream, prm);
}

kda_status kda_prologue(const kda_desc* desc, const kda_prologue_params* prm, const void* q_raw,
                        const void* k_raw, const void* v_raw, const void* g_raw,
                        const void* beta_logit, void* q, void* k, void* v, void* log_alpha,
                        void* beta, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_prologue");
    kda_status st = check_desc(desc, false);
    if (st != KDA_OK) return st;
    if (desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!check_prologue(prm)) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens == 0) return KDA_OK;
    const void* in[5] = {q_raw, k_raw, v_raw, g_raw, beta_logit};
    const void* outs[5] = {q, k, v, log_alpha, beta};
    for (int i = 0; i < 5; ++i) {
        if (!in[i] || !outs[i]) return KDA_ERR_INVALID_ARG;
        if (i < 4 && (!aligned16(in[i]) || !aligned16(outs[i]))) return KDA_ERR_INVALID_ARG;
        for (int j = 0; j < 5; ++j)
            if (outs[i] == in[j] || (j != i && outs[i] == outs[j])) return KDA_ERR_INVALID_ARG;
    }
    cudaError_t e = kda::launch_prologue(desc->total_tokens * desc->num_heads, desc->num_heads,
                                         q_raw, k_raw, v_raw, g_raw, beta_logit, prm->A_log,
                                         prm->dt_bias, prm->lower_bound, prm->q_scale, q, k, v,
                                         log_alpha, beta, (cudaStream_t)stream);
    g_launches += 1;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_prologue_conv(const kda_desc* desc, const kda_prologue_params* prm,
                             const kda_conv_params* conv, const int32_t* cu_seqlens,
                             const void* q_raw, const void* k_raw, const void* v_raw,
                             const void* g_raw, const void* beta_logit, void* q, void* k, void* v,
                             void* log_alpha, void* beta, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_prologue_conv");
    kda_status st = check_desc(desc, true);
    if (st != KDA_OK) return st;
    if (desc->in_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!check_prologue(prm) || !conv || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (!conv->w_q || !conv->w_k || !conv->w_v || !aligned16(conv->w_q) || !aligned16(conv->w_k) ||
        !aligned16(conv->w_v) || !aligned16(conv->cache_in) || !aligned16(conv->cache_out))
        return KDA_ERR_INVALID_ARG;
    const void* in[5] = {q_raw, k_raw, v_raw, g_raw, beta_logit};
    const void* outs[5] = {q, k, v, log_alpha, beta};
    if (desc->total_tokens > 0) {
        for (int i = 0; i < 5; ++i) {
            if (!in[i] || !outs[i]) return KDA_ERR_INVALID_ARG;
            if (i < 4 && (!aligned16(in[i]) || !aligned16(outs[i]))) return KDA_ERR_INVALID_ARG;
            for (int j = 0; j < 5; ++j)
                if (outs[i] == in[j] || (j != i && outs[i] == outs[j])) return KDA_ERR_INVALID_ARG;
        }
    }
    const void* co = conv->cache_out;
    for (int i = 0; i < 5; ++i)
        if (co && (co == in[i] || co == outs[i])) return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_prologue_conv(
        desc->total_tokens * desc->num_heads, desc->num_heads, desc->num_seqs, q_raw, k_raw, v_raw,
        g_raw, beta_logit, prm->A_log, prm->dt_bias, prm->lower_bound, prm->q_scale, conv->w_q,
        conv->w_k, conv->w_v, conv->cache_in, conv->cache_out, cu_seqlens, q, k, v, log_alpha,
        beta, (cudaStream_t)stream);
    g_launches += (desc->total_tokens > 0 ? 1 : 0) + (conv->cache_out ? 1 : 0);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode_step(const kda_desc* desc, const void* q, const void* k, const void* v,
                           const void* log_alpha, const void* beta, float* state, void* out,
                           kda_stream_t stream) {
    NvtxRange nvtx_range("kda_decode_step");
    return decode_step_impl(desc, q, k, v, log_alpha, beta, state, out, stream, nullptr);
}

kda_status kda_decode_step_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                    const void* q_raw, const void* k_raw, const void* v_raw,
                                    const void* g_raw, const void* beta_logit, float* state,
                                    void* out, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_decode_step_prologue");
    if (!prm) return KDA_ERR_INVALID_ARG;
    return decode_step_impl(desc, q_raw, k_raw, v_raw, g_raw, beta_logit, state, out, stream, prm);
}

kda_status kda_decode_window(const kda_desc* desc, const void* q, const void* k, const void* v,
                             const void* log_alpha, const void* beta, const int32_t* cu_seqlens,
                             float* state, void* out, const int32_t* commit, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_decode_window");
    return decode_window_impl(desc, q, k, v, log_alpha, beta, cu_seqlens, state, out, commit,
                              stream, nullptr);
}

kda_status kda_decode_window_prologue(const kda_desc* desc, const kda_prologue_params* prm,
                                      const void* q_raw, const void* k_raw, const void* v_raw,
                                      const void* g_raw, const void* beta_logit,
                                      const int32_t* cu_seqlens, float* state, void* out,
                                      const int32_t* commit, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_decode_window_prologue");
    if (!prm) return KDA_ERR_INVALID_ARG;
    return decode_window_impl(desc, q_raw, k_raw, v_raw, g_raw, beta_logit, cu_seqlens, state,
                              out, commit, stream, prm);
}

size_t kda_bwd_workspace_bytes(const kda_desc* desc) {
    if (check_desc(desc, true) != KDA_OK) return 0;
    const int64_t chunks = kda::backward_chunks(desc->host_seqlens, desc->num_seqs);
    return kda::backward_workspace_floats(desc->num_seqs, desc->num_heads, chunks) * sizeof(float);
}

kda_status kda_bwd(const kda_desc* desc, const void* q, const void* k, const void* v,
                   const void* log_alpha, const void* beta, const float* init_state,
                   const int32_t* cu_seqlens, const float* d_out, const float* d_state, float* dq,
                   float* dk, float* dv, float* dlog_alpha, float* dbeta, float* dinit_state,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    NvtxRange nvtx_range("kda_bwd");
    kda_status st = check_desc(desc, true);
    if (st != KDA_OK) return st;
    if (!cu_seqlens || !dinit_state) return KDA_ERR_INVALID_ARG;
    const void* in[9] = {q, k, v, log_alpha, beta, init_state, d_out, d_state, cu_seqlens};
    const void* outs[6] = {dq, dk, dv, dlog_alpha, dbeta, dinit_state};
    if (desc->total_tokens > 0) {
        for (int i = 0; i < 7; ++i)
            if (i != 5 && !in[i]) return KDA_ERR_INVALID_ARG;
        for (int i = 0; i < 5; ++i)
            if (!outs[i]) return KDA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < 6; ++i) {
        if (outs[i] && !aligned16(outs[i])) return KDA_ERR_INVALID_ARG;
        for (int j = 0; j < 9; ++j)
            if (outs[i] && outs[i] == in[j]) return KDA_ERR_INVALID_ARG;
        for (int j = 0; j < i; ++j)
            if (outs[i] && outs[i] == outs[j]) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned16(init_state) || !aligned16(d_state) || !aligned16(d_out))
        return KDA_ERR_INVALID_ARG;
    // rows are read four channels at a time
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha))
        return KDA_ERR_INVALID_ARG;
    const size_t need = kda_bwd_workspace_bytes(desc);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    cudaError_t e = kda::launch_backward(
        desc->in_dtype, desc->num_seqs, desc->num_heads, q, k, v, log_alpha, beta, cu_seqlens,
        init_state, d_out, d_state, dq, dk, dv, dlog_alpha, dbeta, dinit_state,
        static_cast<float*>(workspace), kda::backward_chunks(desc->host_seqlens, desc->num_seqs),
        desc->total_tokens, status, (cudaStream_t)stream);
    if ((int64_t)desc->num_seqs * desc->num_heads > 0)
        g_launches += desc->total_tokens > 0 ? 4 : 2;   // index, prep, forward, reverse
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_selftest_wait_timeout(kda_stream_t stream) {
    NvtxRange nvtx_range("kda_selftest_wait_timeout");
    int* status = status_word();
    if (!status) return KDA_ERR_CUDA;
    cudaError_t e = kda::launch_wait_selftest(status, (cudaStream_t)stream);
    g_launches += 1;
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_read_device_status(kda_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KDA_ERR_CUDA;
    int* p = status_word();
    if (!p) return KDA_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    return (kda_status)value;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_DECAY_RANGE: return "KDA_ERR_DECAY_RANGE";
    }
    return "KDA_ERR_UNKNOWN";
}

uint64_t kda_launch_count(void) { return g_launches.load(); }

int32_t kda_version(void) { return 2; }

}  // extern "C"
