// kda_host.cu — kda_fwd_chunked_host: the chunked prefill on HOST buffers.
//
// The host-to-device link is the bound of such a call (the kernels need a small fraction of the
// copy time), so the work is cut into token-range parts and three streams overlap the upload of
// part j+1, the kernels of part j and the download of part j-1.  Part j covers tokens
// [b_j, b_{j+1}) of every sequence longer than b_j; the boundaries are multiples of the 64-token
// chunk, chosen so that the parts hold about equal token counts.  A sequence that spans several
// parts carries its fp32 state from one part's kernel to the next through a device array, as a
// caller resuming a prefill from a saved state would.
//
// Device memory comes from the caller's workspace, laid out as
//   [state: N x H x 128 x 128 fp32][cu_seqlens of every part][3 slots x (q, k, v, g, beta, out)]
// with the sequences ordered by decreasing length, so that the sequences still running in part j
// are a prefix of that order and each part's kernel sees contiguous states.
#include <algorithm>
#include <mutex>
#include <numeric>
#include <vector>

#include "kda_common.cuh"

namespace {

constexpr int kDefaultParts = 8;
constexpr int kMaxParts = 64;
constexpr int kSlots = 3;
// Longest span of one sequence inside one part: at or below it the prefill never splits a
// sequence into segments, so the parts need no segment workspace.
constexpr int64_t kMaxSpan = 65536;
constexpr size_t kStateBytes = 128 * 128 * sizeof(float);

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct HostPlan {
    std::vector<int32_t> order;       // sequences by decreasing length (stable)
    std::vector<int64_t> bound;       // part boundaries b_0 = 0 < b_1 < ... (tokens)
    std::vector<int32_t> active;      // sequences in part j (a prefix of `order`)
    std::vector<int64_t> tokens;      // tokens in part j
    std::vector<int64_t> cu_index;    // first entry of part j's cu_seqlens in the cu region
    std::vector<int32_t> cu_host;     // every part's cu_seqlens, concatenated
    int64_t cap_tokens = 0;           // largest part
    size_t row_bytes = 0;             // bytes of one token row of q (= k, g, v, out)
    size_t beta_row_bytes = 0;
    size_t cu_off = 0, slot_off = 0, slot_bytes = 0, total_bytes = 0;
    size_t off_q = 0, off_k = 0, off_v = 0, off_g = 0, off_beta = 0, off_out = 0;
};

int64_t tokens_before(const kda_desc* d, int64_t b) {
    int64_t s = 0;
    for (int32_t n = 0; n < d->num_seqs; ++n) s += std::min<int64_t>(d->host_seqlens[n], b);
    return s;
}

// Part boundaries: b_j is the first chunk multiple at which a planned share of the tokens lies
// before it, no part spans more than kMaxSpan tokens of a sequence, and the last boundary is the
// longest length.  Only the last part's kernels and download are not hidden behind an upload, so
// from four parts on the last part is planned at 1/(4 parts) of the tokens and the others share
// the rest equally; with fewer parts they are equal.
kda_status make_plan(const kda_desc* d, int32_t parts, HostPlan* p) {
    if (parts < 0 || parts > kMaxParts) return KDA_ERR_INVALID_ARG;
    const int want = parts == 0 ? kDefaultParts : parts;
    const int N = d->num_seqs;
    const int64_t T = d->total_tokens;
    int64_t lmax = 0;
    for (int n = 0; n < N; ++n) lmax = std::max<int64_t>(lmax, d->host_seqlens[n]);
    p->order.resize(N);
    std::iota(p->order.begin(), p->order.end(), 0);
    std::stable_sort(p->order.begin(), p->order.end(), [d](int32_t a, int32_t b) {
        return d->host_seqlens[a] > d->host_seqlens[b];
    });
    p->bound.assign(1, 0);
    for (int j = 1; j < want && p->bound.back() < lmax; ++j) {
        // smallest multiple of the chunk above the previous boundary reaching the planned share
        const int64_t num = want >= 4 ? T * j * (4 * want - 1) : T * j;
        const int64_t den = want >= 4 ? (int64_t)(want - 1) * 4 * want : want;
        const int64_t goal = (num + den - 1) / den;
        int64_t lo = p->bound.back() / kda::kChunk + 1, hi = (lmax + kda::kChunk - 1) / kda::kChunk;
        while (lo < hi) {
            const int64_t mid = (lo + hi) / 2;
            if (tokens_before(d, mid * kda::kChunk) >= goal) hi = mid; else lo = mid + 1;
        }
        const int64_t b = lo * kda::kChunk;
        if (b >= lmax) break;
        p->bound.push_back(b);
    }
    p->bound.push_back(std::max<int64_t>(lmax, 0));
    // no part longer than kMaxSpan tokens (kMaxSpan is a multiple of the chunk)
    std::vector<int64_t> fine(1, 0);
    for (size_t j = 1; j < p->bound.size(); ++j) {
        while (p->bound[j] - fine.back() > kMaxSpan) fine.push_back(fine.back() + kMaxSpan);
        if (p->bound[j] > fine.back() || j + 1 == p->bound.size()) fine.push_back(p->bound[j]);
    }
    if (fine.size() < 2) fine.push_back(0);  // every sequence empty: one part of zero tokens
    p->bound.swap(fine);
    const int m = (int)p->bound.size() - 1;
    p->active.resize(m);
    p->tokens.resize(m);
    p->cu_index.resize(m);
    p->cu_host.clear();
    p->cap_tokens = 0;
    for (int j = 0; j < m; ++j) {
        const int64_t b0 = p->bound[j], span = p->bound[j + 1] - b0;
        int a = 0;
        int64_t tok = 0;
        p->cu_index[j] = (int64_t)p->cu_host.size();
        p->cu_host.push_back(0);
        for (int i = 0; i < N; ++i) {
            const int64_t L = d->host_seqlens[p->order[i]];
            if (j > 0 && L <= b0) break;  // sorted: every later sequence has ended too
            tok += std::clamp<int64_t>(L - b0, 0, span);
            p->cu_host.push_back((int32_t)tok);
            ++a;
        }
        p->active[j] = a;
        p->tokens[j] = tok;
        p->cap_tokens = std::max(p->cap_tokens, tok);
    }
    const size_t elt = d->in_dtype == KDA_BF16 ? 2 : 4;
    p->row_bytes = (size_t)d->num_heads * 128 * elt;
    p->beta_row_bytes = (size_t)d->num_heads * elt;
    const size_t cap = (size_t)p->cap_tokens;
    p->cu_off = align256((size_t)N * d->num_heads * kStateBytes);
    p->slot_off = p->cu_off + align256(p->cu_host.size() * sizeof(int32_t));
    p->off_q = 0;
    p->off_k = p->off_q + align256(cap * p->row_bytes);
    p->off_v = p->off_k + align256(cap * p->row_bytes);
    p->off_g = p->off_v + align256(cap * p->row_bytes);
    p->off_beta = p->off_g + align256(cap * p->row_bytes);
    p->off_out = p->off_beta + align256(cap * p->beta_row_bytes);
    p->slot_bytes = p->off_out + align256(cap * p->row_bytes);
    p->total_bytes = p->slot_off + kSlots * p->slot_bytes;
    return KDA_OK;
}

bool check_desc_host(const kda_desc* d) {
    if (!d || !d->host_seqlens || d->num_seqs < 1 || d->num_heads < 1 || d->reserved != 0)
        return false;
    if (d->d_k != 128 || d->d_v != 128) return false;
    if (d->in_dtype != KDA_BF16 && d->in_dtype != KDA_FP32) return false;
    int64_t sum = 0;
    for (int32_t n = 0; n < d->num_seqs; ++n) {
        if (d->host_seqlens[n] < 0) return false;
        sum += d->host_seqlens[n];
    }
    return sum == d->total_tokens && d->total_tokens <= INT32_MAX;
}

// Three non-blocking streams per device, created on first use and kept for the process.
constexpr int kMaxDevices = 64;
cudaStream_t g_streams[kMaxDevices][3] = {};
std::mutex g_streams_mu;

cudaError_t device_streams(cudaStream_t* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_streams_mu);
    for (int i = 0; i < 3; ++i) {
        if (!g_streams[dev][i]) {
            e = cudaStreamCreateWithFlags(&g_streams[dev][i], cudaStreamNonBlocking);
            if (e != cudaSuccess) return e;
        }
        s[i] = g_streams[dev][i];
    }
    return cudaSuccess;
}

// Copy `count` states between the ordered device array and the caller's host array, merging
// runs of consecutive sequence indices into one copy.
cudaError_t copy_states(const HostPlan& p, int heads, int i0, int i1, char* dev_states,
                        char* host_states, cudaMemcpyKind kind, cudaStream_t s) {
    const size_t unit = (size_t)heads * kStateBytes;
    for (int i = i0; i < i1;) {
        int j = i + 1;
        while (j < i1 && p.order[j] == p.order[j - 1] + 1) ++j;
        char* dv = dev_states + (size_t)i * unit;
        char* hv = host_states + (size_t)p.order[i] * unit;
        cudaError_t e = kind == cudaMemcpyHostToDevice
                            ? cudaMemcpyAsync(dv, hv, (size_t)(j - i) * unit, kind, s)
                            : cudaMemcpyAsync(hv, dv, (size_t)(j - i) * unit, kind, s);
        if (e != cudaSuccess) return e;
        i = j;
    }
    return cudaSuccess;
}

// A run of consecutive sequences (in the plan's order) that contribute the same number of rows
// to a part and lie at a constant stride in the caller's arrays: one strided copy per tensor.
struct Run {
    int count;
    int64_t rows, dev_row, host_row, pitch;  // pitch: rows between the sequences' first rows
};

// Strides up to 1 GiB go into one 2D copy; a longer one falls back to a copy per sequence.
constexpr int64_t kMaxPitchBytes = int64_t(1) << 30;

void part_runs(const HostPlan& p, const kda_desc* d, const std::vector<int64_t>& start, int j,
               std::vector<Run>* runs) {
    runs->clear();
    const int64_t b0 = p.bound[j], span = p.bound[j + 1] - b0;
    const int64_t max_pitch = kMaxPitchBytes / (int64_t)p.row_bytes;
    int64_t dev_row = 0;
    for (int i = 0; i < p.active[j]; ++i) {
        const int n = p.order[i];
        const int64_t rows = std::clamp<int64_t>(d->host_seqlens[n] - b0, 0, span);
        if (rows == 0) continue;
        const int64_t host_row = start[n] + b0;
        if (!runs->empty()) {
            Run& r = runs->back();
            const int64_t pitch = host_row - (r.host_row + (r.count - 1) * r.pitch);
            const bool next_to = r.dev_row + r.count * r.rows == dev_row;
            if (rows == r.rows && next_to && pitch >= rows && pitch <= max_pitch &&
                (r.count == 1 || pitch == r.pitch)) {
                r.pitch = pitch;
                r.count += 1;
                dev_row += rows;
                continue;
            }
        }
        runs->push_back(Run{1, rows, dev_row, host_row, rows});
        dev_row += rows;
    }
}

cudaError_t copy_run(const Run& r, size_t rb, char* dev, char* host, cudaMemcpyKind kind,
                     cudaStream_t s) {
    char* dv = dev + (size_t)r.dev_row * rb;
    char* hv = host + (size_t)r.host_row * rb;
    const size_t width = (size_t)r.rows * rb;
    if (r.count == 1)
        return kind == cudaMemcpyHostToDevice ? cudaMemcpyAsync(dv, hv, width, kind, s)
                                              : cudaMemcpyAsync(hv, dv, width, kind, s);
    const size_t hp = (size_t)r.pitch * rb;
    return kind == cudaMemcpyHostToDevice
               ? cudaMemcpy2DAsync(dv, width, hv, hp, width, (size_t)r.count, kind, s)
               : cudaMemcpy2DAsync(hv, hp, dv, width, width, (size_t)r.count, kind, s);
}

struct Events {
    cudaEvent_t ev[1 + 3 * kSlots] = {};
    ~Events() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
    }
    cudaError_t create() {
        for (cudaEvent_t& e : ev) {
            cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
        }
        return cudaSuccess;
    }
    cudaEvent_t start() const { return ev[0]; }
    cudaEvent_t in(int s) const { return ev[1 + s]; }
    cudaEvent_t run(int s) const { return ev[1 + kSlots + s]; }
    cudaEvent_t out(int s) const { return ev[1 + 2 * kSlots + s]; }
};

}  // namespace

extern "C" {

size_t kda_fwd_host_workspace_bytes(const kda_desc* desc, int32_t parts) {
    if (!check_desc_host(desc)) return 0;
    HostPlan p;
    if (make_plan(desc, parts, &p) != KDA_OK) return 0;
    return p.total_bytes;
}

kda_status kda_fwd_chunked_host(const kda_desc* desc, const void* q, const void* k,
                                const void* v, const void* log_alpha, const void* beta,
                                const float* init_state, void* out, float* final_state,
                                int32_t parts, void* workspace, size_t workspace_bytes,
                                kda_stream_t stream) {
    if (!check_desc_host(desc)) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta || !out))
        return KDA_ERR_INVALID_ARG;
    if (out && (out == q || out == k || out == v || out == log_alpha || out == beta))
        return KDA_ERR_INVALID_ARG;
    HostPlan p;
    kda_status st = make_plan(desc, parts, &p);
    if (st != KDA_OK) return st;
    if (!workspace || workspace_bytes < p.total_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KDA_ERR_WORKSPACE;

    cudaStream_t s3[3];
    if (device_streams(s3) != cudaSuccess) return KDA_ERR_CUDA;
    cudaStream_t s_in = s3[0], s_run = s3[1], s_out = s3[2];
    Events ev;
    if (ev.create() != cudaSuccess) return KDA_ERR_CUDA;

    char* ws = static_cast<char*>(workspace);
    char* states = ws;
    int32_t* cu_dev = reinterpret_cast<int32_t*>(ws + p.cu_off);
    const int H = desc->num_heads;
    const int N = desc->num_seqs;
    const int m = (int)p.active.size();
    std::vector<int64_t> start(N + 1, 0);
    for (int n = 0; n < N; ++n) start[n + 1] = start[n] + desc->host_seqlens[n];
    const char* src[5] = {static_cast<const char*>(q), static_cast<const char*>(k),
                          static_cast<const char*>(v), static_cast<const char*>(log_alpha),
                          static_cast<const char*>(beta)};
    const size_t dst_off[5] = {p.off_q, p.off_k, p.off_v, p.off_g, p.off_beta};
    const size_t row[5] = {p.row_bytes, p.row_bytes, p.row_bytes, p.row_bytes, p.beta_row_bytes};

    cudaError_t e = cudaSuccess;
    kda_status result = KDA_OK;
    auto ok = [&](cudaError_t r) {
        if (r != cudaSuccess && e == cudaSuccess) e = r;
        return e == cudaSuccess;
    };
    // everything starts after the work already queued on the caller's stream
    if (ok(cudaEventRecord(ev.start(), (cudaStream_t)stream)))
        for (cudaStream_t s : s3) ok(cudaStreamWaitEvent(s, ev.start(), 0));
    if (e == cudaSuccess)
        ok(cudaMemcpyAsync(cu_dev, p.cu_host.data(), p.cu_host.size() * sizeof(int32_t),
                           cudaMemcpyHostToDevice, s_in));
    if (e == cudaSuccess && init_state)
        ok(copy_states(p, H, 0, N, states, reinterpret_cast<char*>(const_cast<float*>(init_state)),
                       cudaMemcpyHostToDevice, s_in));
    std::vector<int32_t> lens;
    std::vector<Run> runs;
    for (int j = 0; j < m && e == cudaSuccess && result == KDA_OK; ++j) {
        const int s = j % kSlots;
        char* slot = ws + p.slot_off + (size_t)s * p.slot_bytes;
        const int64_t b0 = p.bound[j], span = p.bound[j + 1] - b0;
        // upload: this slot's previous part must have been downloaded
        if (j >= kSlots) ok(cudaStreamWaitEvent(s_in, ev.out(s), 0));
        lens.assign(p.active[j], 0);
        for (int i = 0; i < p.active[j]; ++i)
            lens[i] = (int32_t)std::clamp<int64_t>(desc->host_seqlens[p.order[i]] - b0, 0, span);
        part_runs(p, desc, start, j, &runs);
        for (const Run& r : runs)
            for (int a = 0; a < 5 && e == cudaSuccess; ++a)
                ok(copy_run(r, row[a], slot + dst_off[a], const_cast<char*>(src[a]),
                            cudaMemcpyHostToDevice, s_in));
        ok(cudaEventRecord(ev.in(s), s_in));
        // the kernels of this part, on its own description; the state array is read and written
        // in place (the first part reads the caller's initial states, or zeros)
        ok(cudaStreamWaitEvent(s_run, ev.in(s), 0));
        if (e != cudaSuccess) break;
        kda_desc dj = *desc;
        dj.num_seqs = p.active[j];
        dj.total_tokens = p.tokens[j];
        dj.host_seqlens = lens.data();
        const float* init = (j == 0 && !init_state) ? nullptr : reinterpret_cast<float*>(states);
        result = kda_fwd_chunked(&dj, slot + p.off_q, slot + p.off_k, slot + p.off_v,
                                 slot + p.off_g, slot + p.off_beta, init, cu_dev + p.cu_index[j],
                                 slot + p.off_out, reinterpret_cast<float*>(states), nullptr, 0,
                                 (kda_stream_t)s_run);
        if (result != KDA_OK) break;
        ok(cudaEventRecord(ev.run(s), s_run));
        // download this part's outputs, and the final states of the sequences that end here
        ok(cudaStreamWaitEvent(s_out, ev.run(s), 0));
        for (const Run& r : runs)
            if (e == cudaSuccess)
                ok(copy_run(r, p.row_bytes, slot + p.off_out, static_cast<char*>(out),
                            cudaMemcpyDeviceToHost, s_out));
        int end0 = -1, end1 = -1;
        for (int i = 0; i < p.active[j]; ++i)
            if (desc->host_seqlens[p.order[i]] <= p.bound[j + 1]) {  // ends in this part
                if (end0 < 0) end0 = i;
                end1 = i + 1;
            }
        if (final_state && end0 >= 0 && e == cudaSuccess)
            ok(copy_states(p, H, end0, end1, states, reinterpret_cast<char*>(final_state),
                           cudaMemcpyDeviceToHost, s_out));
        ok(cudaEventRecord(ev.out(s), s_out));
    }
    // the call returns when every copy it issued has finished (also after an error, so that no
    // copy into the caller's buffers outlives the call)
    cudaError_t sync = cudaSuccess;
    for (cudaStream_t s : s3) {
        cudaError_t r = cudaStreamSynchronize(s);
        if (sync == cudaSuccess) sync = r;
    }
    if (result != KDA_OK) return result;
    if (e != cudaSuccess || sync != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
