// Tensor-core (tcgen05/TMEM) chunk scan.  Not yet enabled: tc_supported()
// reports no sizes, so AUTO selects the SIMT kernels.
#include "kda_common.cuh"

namespace kda {

namespace {
__device__ int g_tc_error = 0;
}

bool tc_supported(const kda_dims&) { return false; }

size_t tc_workspace_bytes(const kda_dims&, int) { return 0; }

kda_status tc_fwd(const kda_dims&, const void*, const void*, const void*, const void*,
                  const void*, const float*, void*, float*, void*, cudaStream_t) {
    return KDA_ERR_UNSUPPORTED;
}

kda_status tc_bwd(const kda_dims&, const void*, const void*, const void*, const void*,
                  const void*, const float*, const void*, const float*, void*, void*, void*,
                  void*, void*, float*, void*, cudaStream_t) {
    return KDA_ERR_UNSUPPORTED;
}

kda_status tc_take_error(cudaStream_t s) {
    int err = 0;
    if (cudaMemcpyFromSymbolAsync(&err, g_tc_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (err == 0) return KDA_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    cudaStreamSynchronize(s);
    return KDA_ERR_TIMEOUT;
}

}  // namespace kda
