// Shared device helpers and internal launcher declarations of libkda.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr float kGateFloor = -5.0f;  // g is clamped at -5 before exp

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Round a byte count up to a 256-byte multiple (workspace sub-allocation).
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline kda_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// ---- internal launchers (validated arguments only) ----
kda_status decode_launch(const kda_dims& d, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, float* state, void* o,
                         cudaStream_t s);

size_t simt_workspace_bytes(const kda_dims& d, int for_bwd);
// All fp32 arrays of the SIMT workspace (bwd carve; the forward arrays come
// first, so their addresses are the same in the forward carve).
struct SimtWsPtrs {
    float *W, *U, *Qh, *Kb, *Aqk, *Tm, *gam, *dlt;
    float *hs, *dhs, *ddl, *dQh, *dWm, *dKb, *dgam, *dAqk, *dTv, *dbv, *dqh, *dkh;
};
void simt_ws_ptrs(const kda_dims& d, int for_bwd, void* ws, SimtWsPtrs* out);
// GVA reduction: dq[b,t,h] = sum over the value heads of group h of dqh (fp32);
// with d.qk_l2norm, then mapped from the normalised to the raw q (k, alike).
kda_status group_sum_launch(const kda_dims& d, const float* dqh, const float* dkh,
                            const void* q, const void* k, void* dq, void* dk, cudaStream_t s);
kda_status simt_fwd(const kda_dims& d, const void* q, const void* k, const void* v,
                    const void* g, const void* beta, const float* h0, void* o, float* ht,
                    void* ws, cudaStream_t s);
kda_status simt_bwd(const kda_dims& d, const void* q, const void* k, const void* v,
                    const void* g, const void* beta, const float* h0, const void* dout,
                    const float* dht, void* dq, void* dk, void* dv, void* dg, void* dbeta,
                    float* dh0, void* ws, cudaStream_t s);

// Packed variable-length sequences on the SIMT kernels (B == 1; cu_seqlens
// [nseq + 1] on the device; states [nseq][HV][K][V]).
size_t simt_varlen_workspace_bytes(const kda_dims& d, int nseq, int for_bwd);
kda_status simt_fwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const float* h0, void* o, float* ht, void* ws, cudaStream_t s);
kda_status simt_bwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const float* h0, const void* dout, const float* dht, void* dq,
                           void* dk, void* dv, void* dg, void* dbeta, float* dh0, void* ws,
                           cudaStream_t s);
// Reads and clears the device error word of the SIMT kernels (invalid
// cu_seqlens: KDA_ERR_SHAPE).
kda_status simt_take_error(cudaStream_t s);
// The chunk table of a packed batch (both kernel families): ctab [NT][2] =
// (first token, valid rows) of every chunk slot, sfirst [nseq + 1] = each
// sequence's first slot; an invalid cu_seqlens is recorded for kda_check and
// leaves every sequence without chunks.
kda_status varlen_table_launch(const int* cu, int nseq, int T, int C, int NT, int* ctab,
                               int* sfirst, cudaStream_t s);

bool tc_supported(const kda_dims& d);
size_t tc_workspace_bytes(const kda_dims& d, int for_bwd);
// save: also keep the chunk-start states and delta in a backward-sized
// workspace.  from_saved: the workspace holds a saving forward's results for
// these inputs, so the intra-chunk recompute and the forward state pass are
// skipped.
kda_status tc_fwd(const kda_dims& d, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, const float* h0, void* o, float* ht,
                  void* ws, bool save, cudaStream_t s);
kda_status tc_bwd(const kda_dims& d, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, const float* h0, const void* dout,
                  const float* dht, void* dq, void* dk, void* dv, void* dg, void* dbeta,
                  float* dh0, void* ws, bool from_saved, cudaStream_t s);
// Packed variable-length sequences on the tensor-core kernels (same
// arguments as the SIMT versions; save / from_saved as for tc_fwd / tc_bwd).
size_t tc_varlen_workspace_bytes(const kda_dims& d, int nseq, int for_bwd);
kda_status tc_fwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0, void* o,
                         float* ht, void* ws, bool save, cudaStream_t s);
kda_status tc_bwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0,
                         const void* dout, const float* dht, void* dq, void* dk, void* dv,
                         void* dg, void* dbeta, float* dh0, void* ws, bool from_saved,
                         cudaStream_t s);
// Reads and clears the device error word of the tensor-core kernels.
kda_status tc_take_error(cudaStream_t s);
// Diagnostic: a bounded wait on an mbarrier nothing arrives at, with the given
// limit (cycles); it records KDA_ERR_TIMEOUT for the next kda_check.
kda_status tc_selftest_timeout(long long limit_cycles, cudaStream_t s);

}  // namespace kda
