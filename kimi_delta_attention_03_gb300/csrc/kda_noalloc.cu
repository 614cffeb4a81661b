// kda_noalloc.cu — chunked prefill for callers that cannot allocate device memory.
//
// kda_fwd_chunked takes its scratch (the segment workspace of long sequences) from the caller.
// Some callers have no way to provide it: code that runs where cudaMalloc is off limits (inside
// an allocator or memory-pool callback, a plugin host that forbids device allocation, a
// latency-critical path where an allocation may synchronise the device), or a caller that
// simply has no allocator at hand.  This entry point uses a fixed scratch array that lives in
// the library itself instead.  It allocates nothing and calls no allocating routine.
//
// The array is a file-scope __device__ variable, so every GPU that loads this library holds
// kNoAllocScratchBytes of device memory for it until the process exits.  All calls share it.
#include <mutex>

#include "kda_common.cuh"

namespace {

// Largest segment workspace this entry point can serve (KDA_NOALLOC_SCRATCH_BYTES, 48 MiB).
constexpr size_t kNoAllocScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevicesNA = 64;
void* g_scratch_addr[kMaxDevicesNA] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code the array's name
// only stands in for the device symbol, so its address has to be looked up once per device
// (with that device current).
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNA) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" kda_status kda_fwd_chunked_noalloc(const kda_desc* desc, const void* q, const void* k,
                                              const void* v, const void* log_alpha,
                                              const void* beta, const float* init_state,
                                              const int32_t* cu_seqlens, void* out,
                                              float* final_state, kda_stream_t stream) {
    kda_plan_info plan;
    kda_status st = kda_fwd_plan(desc, &plan);
    if (st != KDA_OK) return st;
    if (plan.workspace_bytes > kNoAllocScratchBytes) return KDA_ERR_WORKSPACE;
    // Resolve the array's address on every call, whether or not this one needs scratch, so
    // that the first call on a device does the lookup and later (possibly captured) calls
    // only read the cached address.
    void* scratch = scratch_address();
    if (!scratch) return KDA_ERR_CUDA;
    if (plan.workspace_bytes == 0)  // nothing is split: no scratch is touched
        return kda_fwd_chunked(desc, q, k, v, log_alpha, beta, init_state, cu_seqlens, out,
                               final_state, nullptr, 0, stream);
    // Every workspace slot that is read is first written by the same call, so the array needs
    // no clearing between calls.
    return kda_fwd_chunked(desc, q, k, v, log_alpha, beta, init_state, cu_seqlens, out,
                           final_state, scratch, kNoAllocScratchBytes, stream);
}
