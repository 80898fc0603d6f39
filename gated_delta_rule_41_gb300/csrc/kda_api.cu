// C ABI of libkda: argument validation and kernel selection.  Every entry
// point validates fully before the first launch, so a rejected call enqueues
// nothing and writes nothing.
#include <stdint.h>

#include "kda_common.cuh"

namespace {

using namespace kda;

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

unsigned elem_bytes(const kda_dims& d) { return d.dtype == KDA_BF16 ? 2u : 4u; }

// Largest B * HV * T the chunk kernels index (per-head token rows times two
// fit a signed 32-bit tile coordinate); a token tensor of that many rows at
// K = 128 in bf16 would already take 256 GB.
constexpr long long kMaxHeadTokens = 1LL << 30;

kda_status check_common(const kda_dims* d, bool need_chunk) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
    if (d->impl != KDA_IMPL_AUTO && d->impl != KDA_IMPL_SIMT && d->impl != KDA_IMPL_TCGEN05)
        return KDA_ERR_INVALID_ARG;
    if (d->B < 0 || d->H <= 0 || d->HV <= 0 || d->K <= 0 || d->V <= 0) return KDA_ERR_SHAPE;
    if (need_chunk && d->T < 0) return KDA_ERR_SHAPE;
    if (d->HV % d->H != 0) return KDA_ERR_SHAPE;
    if (d->K > 128 || d->V > 128) return KDA_ERR_UNSUPPORTED;
    if ((long long)d->B * d->HV > 65535) return KDA_ERR_UNSUPPORTED;
    if (need_chunk) {
        const int c = d->chunk_size;
        if (c != 16 && c != 32 && c != 64 && c != 128) return KDA_ERR_UNSUPPORTED;
        if (d->T % c != 0) return KDA_ERR_SHAPE;
        // tile coordinates and row indices are 32-bit: the chunk-start state
        // rows of all heads (2 B HV T at chunk 64) stay below 2^31
        if ((long long)d->B * d->HV * d->T >= kMaxHeadTokens) return KDA_ERR_UNSUPPORTED;
    }
    return KDA_OK;
}

// The SIMT kernels tile K across 256 threads: K must divide 256.
bool simt_supported(const kda_dims& d) { return 256 % d.K == 0; }

// Resolves AUTO; returns KDA_IMPL_SIMT or KDA_IMPL_TCGEN05, or -1 if neither fits.
int pick_impl(const kda_dims& d) {
    if (d.impl == KDA_IMPL_TCGEN05) return tc_supported(d) ? KDA_IMPL_TCGEN05 : -1;
    if (d.impl == KDA_IMPL_SIMT) return simt_supported(d) ? KDA_IMPL_SIMT : -1;
    if (tc_supported(d)) return KDA_IMPL_TCGEN05;
    return simt_supported(d) ? KDA_IMPL_SIMT : -1;
}

// `required` pointers may be null only when the tensors are empty (`empty`);
// every non-null pointer must be aligned to `align` bytes.
kda_status check_ptrs(bool empty, unsigned align, std::initializer_list<const void*> required,
                      std::initializer_list<const void*> optional) {
    for (const void* p : required) {
        if (!p && !empty) return KDA_ERR_INVALID_ARG;
        if (!aligned(p, align)) return KDA_ERR_ALIGNMENT;
    }
    for (const void* p : optional)
        if (p && !aligned(p, align)) return KDA_ERR_ALIGNMENT;
    return KDA_OK;
}

// Alignment the chunk kernels need: the tensor-core path moves tiles with TMA
// and 128-bit accesses (16 bytes); the SIMT path reads elements.
unsigned chunk_align(const kda_dims& d, int impl) {
    return impl == KDA_IMPL_TCGEN05 ? 16u : elem_bytes(d);
}

size_t ws_bytes(const kda_dims& d, int impl, int for_bwd) {
    return impl == KDA_IMPL_TCGEN05 ? tc_workspace_bytes(d, for_bwd)
                                    : simt_workspace_bytes(d, for_bwd);
}

kda_status check_ws(const kda_dims& d, int impl, int for_bwd, const void* ws, size_t bytes) {
    const size_t need = ws_bytes(d, impl, for_bwd);
    if (need == 0) return KDA_OK;
    if (!ws || bytes < need) return KDA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KDA_ERR_ALIGNMENT;
    return KDA_OK;
}

// Empty sequence (T == 0): the final state is the initial one, and the
// gradient of h0 is the upstream gradient of the final state.
kda_status copy_or_zero(const kda_dims& d, float* dst, const float* src, cudaStream_t s) {
    if (!dst) return KDA_OK;
    const size_t bytes = (size_t)d.B * d.HV * d.K * d.V * sizeof(float);
    const cudaError_t e = src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s)
                              : cudaMemsetAsync(dst, 0, bytes, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Variable-length batches: dims as for kda_chunk_fwd except B == 1 and no
// T % chunk_size rule.
kda_status check_varlen_dims(const kda_dims* d, int nseq) {
    if (!d) return KDA_ERR_INVALID_ARG;
    kda_dims t = *d;
    t.T = 0;   // T % chunk_size does not apply
    kda_status st = check_common(&t, true);
    if (st != KDA_OK) return st;
    if (d->T < 0 || d->B != 1 || nseq < 1) return KDA_ERR_SHAPE;
    if ((long long)nseq * d->HV > 65535) return KDA_ERR_UNSUPPORTED;
    // the kernels see the padded chunk slots: ceil(T / C) + nseq of them
    const long long slots = ((long long)d->T + d->chunk_size - 1) / d->chunk_size + nseq;
    if (slots * d->chunk_size * d->HV >= kMaxHeadTokens) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// The kernels of a packed batch: as pick_impl; an empty batch (T == 0) runs
// the SIMT kernels (the tensor maps need rows).
int pick_varlen_impl(const kda_dims& d) {
    const int impl = pick_impl(d);
    if (impl == KDA_IMPL_TCGEN05 && d.T == 0)
        return d.impl == KDA_IMPL_TCGEN05 || !simt_supported(d) ? -1 : KDA_IMPL_SIMT;
    return impl;
}
size_t varlen_ws_bytes(const kda_dims& d, int impl, int nseq, int for_bwd) {
    return impl == KDA_IMPL_TCGEN05 ? tc_varlen_workspace_bytes(d, nseq, for_bwd)
                                    : simt_varlen_workspace_bytes(d, nseq, for_bwd);
}

kda_status check_varlen(const kda_dims* d, const int* cu, int nseq) {
    const kda_status st = check_varlen_dims(d, nseq);
    if (st != KDA_OK) return st;
    if (!cu) return KDA_ERR_INVALID_ARG;
    if (!aligned(cu, 4)) return KDA_ERR_ALIGNMENT;
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_chunk_workspace_bytes(const kda_dims* d, int for_bwd) {
    if (check_common(d, true) != KDA_OK) return 0;
    const int impl = pick_impl(*d);
    if (impl < 0) return 0;
    return ws_bytes(*d, impl, for_bwd ? 1 : 0);
}

static kda_status chunk_fwd(const kda_dims* d, const void* q, const void* k, const void* v,
                            const void* g, const void* beta, const float* h0, void* o,
                            int output_final_state, float* ht, void* workspace,
                            size_t workspace_bytes, void* stream, bool save) {
    kda_status st = check_common(d, true);
    if (st != KDA_OK) return st;
    const int impl = pick_impl(*d);
    if (impl < 0) return KDA_ERR_UNSUPPORTED;
    if (output_final_state && !ht && d->B > 0) return KDA_ERR_INVALID_ARG;
    const bool empty = d->B == 0 || d->T == 0;
    if ((st = check_ptrs(empty, chunk_align(*d, impl), {q, k, v, g, o},
                         {h0, output_final_state ? ht : nullptr})) != KDA_OK)
        return st;
    if ((st = check_ptrs(empty, elem_bytes(*d), {beta}, {})) != KDA_OK)
        return st;
    if ((st = check_ws(*d, impl, save ? 1 : 0, workspace, workspace_bytes)) != KDA_OK) return st;
    float* ht_out = output_final_state ? ht : nullptr;
    auto s = static_cast<cudaStream_t>(stream);
    if (d->B == 0) return KDA_OK;
    if (d->T == 0) return copy_or_zero(*d, ht_out, h0, s);
    if (impl == KDA_IMPL_TCGEN05)
        return tc_fwd(*d, q, k, v, g, beta, h0, o, ht_out, workspace, save, s);
    // the SIMT backward recomputes everything: nothing extra to save
    return simt_fwd(*d, q, k, v, g, beta, h0, o, ht_out, workspace, s);
}

static kda_status chunk_bwd(const kda_dims* d, const void* q, const void* k, const void* v,
                            const void* g, const void* beta, const float* h0, const void* dout,
                            const float* dht, void* dq, void* dk, void* dv, void* dg,
                            void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                            void* stream, bool from_saved) {
    kda_status st = check_common(d, true);
    if (st != KDA_OK) return st;
    const int impl = pick_impl(*d);
    if (impl < 0) return KDA_ERR_UNSUPPORTED;
    const bool empty = d->B == 0 || d->T == 0;
    if ((st = check_ptrs(empty, chunk_align(*d, impl), {q, k, v, g, dout, dq, dk, dv, dg},
                         {h0, dht, dh0})) != KDA_OK)
        return st;
    if ((st = check_ptrs(empty, elem_bytes(*d), {beta, dbeta}, {})) != KDA_OK)
        return st;
    if ((st = check_ws(*d, impl, 1, workspace, workspace_bytes)) != KDA_OK) return st;
    auto s = static_cast<cudaStream_t>(stream);
    if (d->B == 0) return KDA_OK;
    if (d->T == 0) return copy_or_zero(*d, dh0, dht, s);
    if (impl == KDA_IMPL_TCGEN05)
        return tc_bwd(*d, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                      from_saved, s);
    return simt_bwd(*d, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                    s);
}

kda_status kda_chunk_fwd(const kda_dims* d, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, void* o,
                         int output_final_state, float* ht, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return chunk_fwd(d, q, k, v, g, beta, h0, o, output_final_state, ht, workspace,
                     workspace_bytes, stream, false);
}

kda_status kda_chunk_fwd_save(const kda_dims* d, const void* q, const void* k, const void* v,
                              const void* g, const void* beta, const float* h0, void* o,
                              int output_final_state, float* ht, void* workspace,
                              size_t workspace_bytes, void* stream) {
    return chunk_fwd(d, q, k, v, g, beta, h0, o, output_final_state, ht, workspace,
                     workspace_bytes, stream, true);
}

kda_status kda_chunk_bwd(const kda_dims* d, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, const void* dout,
                         const float* dht, void* dq, void* dk, void* dv, void* dg,
                         void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                         void* stream) {
    return chunk_bwd(d, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                     workspace_bytes, stream, false);
}

kda_status kda_chunk_bwd_saved(const kda_dims* d, const void* q, const void* k, const void* v,
                               const void* g, const void* beta, const float* h0,
                               const void* dout, const float* dht, void* dq, void* dk, void* dv,
                               void* dg, void* dbeta, float* dh0, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return chunk_bwd(d, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, workspace,
                     workspace_bytes, stream, true);
}

size_t kda_chunk_workspace_bytes_varlen(const kda_dims* d, int num_seqs, int for_bwd) {
    if (check_varlen_dims(d, num_seqs) != KDA_OK) return 0;
    const int impl = pick_varlen_impl(*d);
    if (impl < 0) return 0;
    return varlen_ws_bytes(*d, impl, num_seqs, for_bwd ? 1 : 0);
}

static kda_status varlen_fwd(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                             const void* q, const void* k, const void* v, const void* g,
                             const void* beta, const float* h0, void* o, int output_final_state,
                             float* ht, void* workspace, size_t workspace_bytes, void* stream,
                             bool save) {
    kda_status st = check_varlen(d, cu_seqlens, num_seqs);
    if (st != KDA_OK) return st;
    const int impl = pick_varlen_impl(*d);
    if (impl < 0) return KDA_ERR_UNSUPPORTED;
    if (output_final_state && !ht) return KDA_ERR_INVALID_ARG;
    const bool empty = d->T == 0;
    if ((st = check_ptrs(empty, chunk_align(*d, impl), {q, k, v, g, o},
                         {h0, output_final_state ? ht : nullptr})) != KDA_OK)
        return st;
    if ((st = check_ptrs(empty, elem_bytes(*d), {beta}, {})) != KDA_OK) return st;
    const size_t need = varlen_ws_bytes(*d, impl, num_seqs, save ? 1 : 0);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_ALIGNMENT;
    auto s = static_cast<cudaStream_t>(stream);
    if (impl == KDA_IMPL_TCGEN05)
        return tc_fwd_varlen(*d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, o,
                             output_final_state ? ht : nullptr, workspace, save, s);
    // the SIMT backward recomputes everything: nothing extra to save
    return simt_fwd_varlen(*d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, o,
                           output_final_state ? ht : nullptr, workspace, s);
}

static kda_status varlen_bwd(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                             const void* q, const void* k, const void* v, const void* g,
                             const void* beta, const float* h0, const void* dout,
                             const float* dht, void* dq, void* dk, void* dv, void* dg,
                             void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                             void* stream, bool from_saved) {
    kda_status st = check_varlen(d, cu_seqlens, num_seqs);
    if (st != KDA_OK) return st;
    const int impl = pick_varlen_impl(*d);
    if (impl < 0) return KDA_ERR_UNSUPPORTED;
    const bool empty = d->T == 0;
    if ((st = check_ptrs(empty, chunk_align(*d, impl), {q, k, v, g, dout, dq, dk, dv, dg},
                         {h0, dht, dh0})) != KDA_OK)
        return st;
    if ((st = check_ptrs(empty, elem_bytes(*d), {beta, dbeta}, {})) != KDA_OK) return st;
    const size_t need = varlen_ws_bytes(*d, impl, num_seqs, 1);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_ALIGNMENT;
    auto s = static_cast<cudaStream_t>(stream);
    if (impl == KDA_IMPL_TCGEN05)
        return tc_bwd_varlen(*d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, dout, dht, dq, dk,
                             dv, dg, dbeta, dh0, workspace, from_saved, s);
    return simt_bwd_varlen(*d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, dout, dht, dq, dk, dv,
                           dg, dbeta, dh0, workspace, s);
}

kda_status kda_chunk_fwd_varlen(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                                const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* h0, void* o,
                                int output_final_state, float* ht, void* workspace,
                                size_t workspace_bytes, void* stream) {
    return varlen_fwd(d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, o, output_final_state, ht,
                      workspace, workspace_bytes, stream, false);
}

kda_status kda_chunk_fwd_varlen_save(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* h0, void* o,
                                     int output_final_state, float* ht, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    return varlen_fwd(d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, o, output_final_state, ht,
                      workspace, workspace_bytes, stream, true);
}

kda_status kda_chunk_bwd_varlen(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                                const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* h0, const void* dout,
                                const float* dht, void* dq, void* dk, void* dv, void* dg,
                                void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                                void* stream) {
    return varlen_bwd(d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg,
                      dbeta, dh0, workspace, workspace_bytes, stream, false);
}

kda_status kda_chunk_bwd_varlen_saved(const kda_dims* d, const int* cu_seqlens, int num_seqs,
                                      const void* q, const void* k, const void* v, const void* g,
                                      const void* beta, const float* h0, const void* dout,
                                      const float* dht, void* dq, void* dk, void* dv, void* dg,
                                      void* dbeta, float* dh0, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    return varlen_bwd(d, cu_seqlens, num_seqs, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg,
                      dbeta, dh0, workspace, workspace_bytes, stream, true);
}

kda_status kda_recurrent_step(const kda_dims* d, const void* q, const void* k, const void* v,
                              const void* g, const void* beta, float* state, void* o,
                              void* stream) {
    kda_status st = check_common(d, false);
    if (st != KDA_OK) return st;
    // the state is streamed with 128-bit accesses; the token vectors by element
    if ((st = check_ptrs(d->B == 0, 16u, {state}, {})) != KDA_OK) return st;
    if ((st = check_ptrs(d->B == 0, elem_bytes(*d), {q, k, v, g, beta, o}, {})) != KDA_OK)
        return st;
    if (d->B == 0) return KDA_OK;
    return decode_launch(*d, q, k, v, g, beta, state, o, static_cast<cudaStream_t>(stream));
}

kda_status kda_check(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    kda_status st = tc_take_error(static_cast<cudaStream_t>(stream));
    if (st != KDA_OK) return st;
    if ((st = simt_take_error(static_cast<cudaStream_t>(stream))) != KDA_OK) return st;
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_selftest_wait_timeout(long long limit_cycles, void* stream) {
    if (limit_cycles < 0 || limit_cycles > 4000000000LL) return KDA_ERR_INVALID_ARG;
    return tc_selftest_timeout(limit_cycles, static_cast<cudaStream_t>(stream));
}

const char* kda_status_str(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_SHAPE: return "invalid shape";
        case KDA_ERR_UNSUPPORTED: return "unsupported sizes, dtype or implementation";
        case KDA_ERR_ALIGNMENT: return "pointer not aligned";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int kda_version(void) { return 10000; }

}  // extern "C"
