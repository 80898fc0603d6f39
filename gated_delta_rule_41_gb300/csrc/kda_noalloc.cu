// Allocation-free chunked forward.
//
// Some callers cannot allocate device memory at the point where they run the
// scan. Examples: code running while a CUDA graph is being captured (a
// cudaMalloc there breaks or is refused by the capture); runtimes that
// hand out memory only from a fixed pool reserved at start-up; and hosts that
// forbid allocation on the step path to keep latency predictable.
// kda_chunk_fwd_noalloc serves them: it runs the SIMT chunked forward with
// its scratch in a file-scope device array instead of a caller-provided
// workspace.
#include <mutex>

#include "kda_common.cuh"

namespace kda {
namespace {

// Largest scratch the allocation-free forward may use (32 MiB).  The array
// below lives in every GPU that loads the library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 64;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Host code may
// not use the array's name as a device pointer, so it is looked up once per
// device (with that device current) and cached.
kda_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KDA_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_chunk_fwd_noalloc(const kda_dims* dims, const void* q, const void* k,
                                            const void* v, const void* g, const void* beta,
                                            const float* h0, void* o, int output_final_state,
                                            float* ht, void* stream) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    kda_dims d = *dims;
    d.impl = KDA_IMPL_SIMT;
    const size_t need = kda_chunk_workspace_bytes(&d, 0);
    if (need > kda::kNoAllocScratchBytes) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        const kda_status st = kda::scratch_address(&scratch);
        if (st != KDA_OK) return st;
    }
    // need == 0 means invalid dims (or an empty problem): kda_chunk_fwd reports it.
    return kda_chunk_fwd(&d, q, k, v, g, beta, h0, o, output_final_state, ht, scratch, need,
                         stream);
}
