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
// not use the array's name as a device pointer, so the address comes from
// cudaGetSymbolAddress with the device current.  Outside stream capture it is
// looked up again on every call (cheap once the module is loaded), so a
// device reset that reloads the module at another address is picked up.
// While `stream` is being captured the address cached by the last call made
// outside capture on this device is used; without one the call fails.
kda_status scratch_address(cudaStream_t stream, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KDA_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KDA_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    } else if (!g_noalloc_addr[dev]) {
        return KDA_ERR_CUDA;
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
    // Every call that gets this far looks the address up (also an empty
    // problem), so any such call made before a capture serves as its set-up.
    void* scratch = nullptr;
    const kda_status st = kda::scratch_address(static_cast<cudaStream_t>(stream), &scratch);
    if (st != KDA_OK) return st;
    // need == 0 means invalid dims (or an empty problem): kda_chunk_fwd reports it.
    return kda_chunk_fwd(&d, q, k, v, g, beta, h0, o, output_final_state, ht,
                         need > 0 ? scratch : nullptr, need, stream);
}
