/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) chunk scan and
 * single-token decode step, hand-written CUDA for sm_103a (GB300).
 *
 * The operation (per batch b and value head hv, state S of K x V floats):
 *
 *     a_t = exp(max(g_t, -5))                 per key channel
 *     e_t = v_t - (diag(a_t) S_{t-1})^T k_t   the key reads the decayed state
 *     S_t = diag(a_t) S_{t-1} + beta_t k_t e_t^T
 *     o_t = S_t^T (scale * q_t)               the query reads the updated state
 *
 * Defined by "KDA 训练 → 推理 手写实现" (K3 README), table 实现路线表, row L1
 * (recurrence), row L2 (chunk form: in-chunk cumsum of g, lower-triangular
 * system, triangular solve, state passing between chunks), row L6 (decode
 * state [B,HV,K,V]); its table 关键约束 / 风险点 fixes GVA (value head hv
 * reads key head hv / (HV/H), dq/dk summed back over the group), scale
 * 1/sqrt(K) applied to q at entry, the clamp of g at -5 before exp, and
 * chunk_size 64 with T % chunk_size == 0.  The "KDA CUDA Trainer" README
 * (section on the mixing module) fixes the order: decay, delta write, read.
 *
 * Conventions for every entry point
 * ---------------------------------
 * Layout   All tensors are dense, row-major, contiguous:
 *            q, k  [B,T,H,K]    v, o, do  [B,T,HV,V]    g  [B,T,HV,K]
 *            beta  [B,T,HV]     states (h0, ht, dht, dh0, decode state) [B,HV,K,V]
 *          Gradients have the shape of the input they belong to (dq, dk at
 *          H heads; dv, dg, dbeta at HV heads).
 * Dtypes   q, k, v, g, beta, o and all gradients of those are `dtype`
 *          (KDA_F32 or KDA_BF16).  States are always float32.
 * Memory   Every pointer is a DEVICE pointer.  The caller owns every buffer,
 *          including the workspace.  The library never allocates device
 *          memory, frees or synchronises inside these calls; all work is
 *          ordered on `stream` (a cudaStream_t; NULL = legacy default
 *          stream).  One exception to "enqueued on `stream`": a stateless
 *          tensor-core backward without dht runs its reverse state pass on a
 *          second stream that the library creates once per device.  That
 *          stream waits for `stream` first, and `stream` waits for it (CUDA
 *          events made for the call) before the call's later kernels, so
 *          callers see only `stream`'s order.
 * Alignment  Every pointer must be aligned to its element size.  In addition:
 *          the decode state must be 16-byte aligned; with the tensor-core
 *          implementation q, k, v, g, o, dout, dq, dk, dv, dg, h0, ht, dht
 *          and dh0 must be 16-byte aligned; the workspace 256-byte aligned.
 * Gates    g is a log-decay: values <= 0 are the supported domain (values
 *          below -5 are clamped to -5; positive values may overflow the
 *          in-chunk decay factors and are not supported).
 * Sizes    B * HV * T must stay below 2^30 (for packed sequences: the padded
 *          slot count (ceil(T / chunk_size) + num_seqs) * chunk_size * HV),
 *          and B * HV at most 65535; larger problems are refused with
 *          KDA_ERR_UNSUPPORTED.  Tile coordinates and row indices are 32-bit.
 *          A token tensor at the first limit would hold 256 GB at K = 128.
 * Errors   Arguments are validated before any launch; on a validation error
 *          nothing is enqueued and no output is written.  KDA_ERR_CUDA means
 *          a launch failed (cudaGetLastError); KDA_ERR_TIMEOUT means a device
 *          wait gave up (reported by kda_check).
 * Threads  Calls are thread-safe; calls on different streams may overlap if
 *          they use distinct outputs and workspaces.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer where one is required, bad flag */
    KDA_ERR_SHAPE = 2,        /* non-positive size, HV % H != 0, T % chunk != 0 */
    KDA_ERR_UNSUPPORTED = 3,  /* K or V > 128, chunk not in {16,32,64,128}, impl not
                                 available for these sizes or this dtype */
    KDA_ERR_ALIGNMENT = 4,    /* a pointer is misaligned (see Alignment above) */
    KDA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
    KDA_ERR_CUDA = 6,         /* a CUDA launch or runtime call failed */
    KDA_ERR_TIMEOUT = 7       /* a bounded device wait expired */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Which kernel family runs the chunk scan.
 *   KDA_IMPL_AUTO     tensor-core path when it supports the sizes, else SIMT.
 *   KDA_IMPL_SIMT     fp32 CUDA-core kernels; any K, V <= 128, chunk 16/32/64
 *                     or 128, f32 or bf16 inputs.  At chunk 128 a chunk's
 *                     C x C matrices live in the workspace, not in shared
 *                     memory (a slower tile configuration).
 *   KDA_IMPL_TCGEN05  tcgen05/TMEM tensor-core kernels; bf16, K = V = 128 or
 *                     K = V = 64 (run at 128 with the upper channels zero),
 *                     chunk 64.  KDA_ERR_UNSUPPORTED otherwise.  With
 *                     dht != NULL the tensor-core backward runs a two-term
 *                     variant: an O(1) final-state gradient makes the
 *                     products of the state gradient with delta and Kb cancel
 *                     to values far below their terms, so U, Kb, delta and
 *                     the state gradient also leave their kernels as bf16 low
 *                     parts (x - bf16(x)) and those products take three terms
 *                     (hi hi + lo hi + hi lo). */
typedef enum { KDA_IMPL_AUTO = 0, KDA_IMPL_SIMT = 1, KDA_IMPL_TCGEN05 = 2 } kda_impl;

typedef struct {
    int B, T, H, HV, K, V;
    int chunk_size;   /* 16, 32, 64 or 128 (128: the SIMT kernels only; AUTO picks them);
                       * T % chunk_size == 0 (ignored by the decode step) */
    float scale;      /* multiplies q; pass 1/sqrt(K) for the standard scale */
    kda_dtype dtype;
    kda_impl impl;
    /* Nonzero: the kernels L2-normalise q and k over K, per token and head,
     * before use: x_n = x / max(||x||_2, 1e-12), in fp32 (the "q/k L2-norm"
     * variant of the K3 README's test-status table, row L3/L4).  Results are
     * those of the scan on the normalised q, k; dq and dk are the gradients
     * with respect to the raw q, k: dx = (dx_n - x_n <x_n, dx_n>) / max(||x||, 1e-12).
     * Zero: q and k are used as given (a caller that normalises them itself). */
    int qk_l2norm;
} kda_dims;

/* Bytes of device workspace that kda_chunk_fwd (for_bwd = 0) or
 * kda_chunk_bwd (for_bwd = 1) needs for these dims; 0 on invalid dims.
 * The workspace must be 256-byte aligned and need not be zeroed. */
size_t kda_chunk_workspace_bytes(const kda_dims* dims, int for_bwd);

/* Chunked forward scan (K3 row L2; row L1 semantics).
 *   h0                 initial state [B,HV,K,V] f32, or NULL for zeros.
 *   o                  output [B,T,HV,V] (dtype).
 *   output_final_state nonzero: write the state after token T-1 to ht.
 *   ht                 [B,HV,K,V] f32; required iff output_final_state. */
kda_status kda_chunk_fwd(const kda_dims* dims, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, void* o,
                         int output_final_state, float* ht, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Backward of kda_chunk_fwd (K3 row L4 role: dq, dk, dv, dg, dbeta).
 * Stateless: it recomputes the forward from the inputs.  On the tensor cores
 * without dht the recomputed forward state pass and the reverse state pass
 * run side by side (the reverse pass needs only dout and the intra-chunk
 * quantities), the latter on the library's second stream (see Memory).
 *   dout   upstream gradient of o [B,T,HV,V] (dtype).
 *   dht    upstream gradient of the final state [B,HV,K,V] f32, or NULL.
 *   dq, dk [B,T,H,K]; dv [B,T,HV,V]; dg [B,T,HV,K]; dbeta [B,T,HV] (dtype).
 *   dh0    gradient of h0 [B,HV,K,V] f32, or NULL to skip.
 * dg is zero where g < -5 (the clamp); g == -5 passes the gradient. */
kda_status kda_chunk_bwd(const kda_dims* dims, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, const void* dout,
                         const float* dht, void* dq, void* dk, void* dv, void* dg,
                         void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Forward that also keeps in the workspace what the backward needs, the way
 * an autograd function saves tensors for its backward pass: the intra-chunk
 * operands (W, U, decayed q and k, Aqk, T), the chunk decays, and the state at
 * every chunk start with each chunk's delta.  Arguments and results are
 * those of kda_chunk_fwd, but the workspace must hold
 * kda_chunk_workspace_bytes(dims, 1) bytes.  Hand that workspace, untouched,
 * to kda_chunk_bwd_saved.  With the SIMT kernels it runs the plain forward
 * (their backward recomputes). */
kda_status kda_chunk_fwd_save(const kda_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* beta, const float* h0,
                              void* o, int output_final_state, float* ht, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Backward from a workspace filled by kda_chunk_fwd_save with the same dims
 * (impl included), inputs and h0, and not written since.  Arguments, results
 * and errors are those of kda_chunk_bwd.  The tensor-core kernels skip the
 * intra-chunk recompute and the forward state pass unless dht is given (their
 * two-term variant recomputes: the saving forward keeps no low parts); a call
 * that recomputes (that one, or any call on the SIMT kernels) reads nothing
 * saved from the workspace, so its results do not depend on what it holds.  A
 * workspace not filled as stated gives undefined results, not an error. */
kda_status kda_chunk_bwd_saved(const kda_dims* dims, const void* q, const void* k,
                               const void* v, const void* g, const void* beta, const float* h0,
                               const void* dout, const float* dht, void* dq, void* dk, void* dv,
                               void* dg, void* dbeta, float* dh0, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Packed variable-length sequences.  The pages run one length per batch
 * (the DM-KDAGQA-1.7B-SD card notes that its KDA layers have no padding
 * mask); these entry points let a batch of unequal sequences be packed
 * along T instead, each sequence scanned on its own.
 *   dims        B must be 1; T = the total token count (any T >= 0, no
 *               multiple of chunk_size needed); impl as for kda_chunk_fwd
 *               (AUTO: the tensor cores for bf16, K = V = 64 or 128, chunk
 *               64, and T > 0; else the SIMT kernels).  On the tensor cores
 *               each sequence's chunks are tiles of 64 tokens from its
 *               first token; the state passes run one CTA per (sequence,
 *               value head).  The backward always recomputes the forward.
 *   cu_seqlens  DEVICE int32 [num_seqs + 1]: sequence s is tokens
 *               [cu_seqlens[s], cu_seqlens[s+1]); it must start at 0, end at
 *               T and not decrease (empty sequences allowed).  It is read on
 *               the device only; a violation is reported by kda_check as
 *               KDA_ERR_SHAPE, and then no sequence is scanned (the final
 *               states are the initial ones, o is not written) and nothing is
 *               accessed out of bounds.
 *   h0, ht, dht, dh0  per sequence: [num_seqs][HV][K][V] f32.
 *   Other arguments, layouts and results are those of kda_chunk_fwd /
 *   kda_chunk_bwd with B = 1, and the workspace must hold
 *   kda_chunk_workspace_bytes_varlen bytes (0 on invalid dims).  Each
 *   sequence's last chunk may be partial: its rows past the sequence end enter
 *   as q = k = v = 0, g = 0, beta = 0 (which leaves the state unchanged) and
 *   are not written. */
size_t kda_chunk_workspace_bytes_varlen(const kda_dims* dims, int num_seqs, int for_bwd);
kda_status kda_chunk_fwd_varlen(const kda_dims* dims, const int* cu_seqlens, int num_seqs,
                                const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* h0, void* o,
                                int output_final_state, float* ht, void* workspace,
                                size_t workspace_bytes, void* stream);
kda_status kda_chunk_bwd_varlen(const kda_dims* dims, const int* cu_seqlens, int num_seqs,
                                const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* h0, const void* dout,
                                const float* dht, void* dq, void* dk, void* dv, void* dg,
                                void* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                                void* stream);

/* The saving pair of the packed entry points, as kda_chunk_fwd_save /
 * kda_chunk_bwd_saved are of the fixed-length ones: the forward keeps what
 * the backward needs in a workspace of kda_chunk_workspace_bytes_varlen(dims,
 * num_seqs, 1) bytes, and the backward, given that workspace untouched and
 * the same dims, cu_seqlens and inputs, skips the intra-chunk recompute and
 * the forward state pass on the tensor cores (unless dht is given; the SIMT
 * kernels always recompute).  Arguments, results and errors otherwise as
 * kda_chunk_fwd_varlen / kda_chunk_bwd_varlen. */
kda_status kda_chunk_fwd_varlen_save(const kda_dims* dims, const int* cu_seqlens, int num_seqs,
                                     const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* h0, void* o,
                                     int output_final_state, float* ht, void* workspace,
                                     size_t workspace_bytes, void* stream);
kda_status kda_chunk_bwd_varlen_saved(const kda_dims* dims, const int* cu_seqlens, int num_seqs,
                                      const void* q, const void* k, const void* v, const void* g,
                                      const void* beta, const float* h0, const void* dout,
                                      const float* dht, void* dq, void* dk, void* dv, void* dg,
                                      void* dbeta, float* dh0, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* One decode token per head, state updated in place (K3 row L6).
 * dims->T is ignored; q, k [B,H,K]; v, o [B,HV,V]; g [B,HV,K]; beta [B,HV]
 * (dtype); state [B,HV,K,V] f32, read and overwritten. */
kda_status kda_recurrent_step(const kda_dims* dims, const void* q, const void* k,
                              const void* v, const void* g, const void* beta, float* state,
                              void* o, void* stream);

/* Allocation-free variant of kda_chunk_fwd, for callers that cannot
 * allocate device memory where they run the scan: code running while a CUDA
 * graph is captured, runtimes that only hand out memory from a pool fixed at
 * start-up, or step loops that forbid allocation.  (The pages describe no
 * such entry point; it is an addition of this library.)
 *   Arguments and results are those of kda_chunk_fwd without the workspace;
 *   dims->impl is ignored and the SIMT kernels run.  Their scratch lives in a
 *   file-scope device array of 32 MiB that every GPU loading the library
 *   keeps until the process exits.  The scratch a call needs is
 *   kda_chunk_workspace_bytes of the same dims with impl = KDA_IMPL_SIMT and
 *   for_bwd = 0; calls that need more than 32 MiB are rejected with
 *   KDA_ERR_WORKSPACE before anything is enqueued.
 *   The function calls no cudaMalloc, cudaFree or allocating library routine.
 *   It finds the array's device address with cudaGetSymbolAddress (with the
 *   calling device current) on every call made outside stream capture, so a
 *   device reset is picked up; a call made while `stream` is captured uses
 *   the address found by the last call outside capture on that device, and
 *   fails with KDA_ERR_CUDA if there was none.  Any call that passes the
 *   size check (an empty problem included) does that look-up: make one on
 *   each device before capturing.  Every call shares the one array and
 *   nothing in it needs to start at zero; calls whose work overlaps on the
 *   GPU (several streams, several host threads) race on it, so serialise
 *   them. */
kda_status kda_chunk_fwd_noalloc(const kda_dims* dims, const void* q, const void* k,
                                 const void* v, const void* g, const void* beta, const float* h0,
                                 void* o, int output_final_state, float* ht, void* stream);

/* Synchronise `stream`, then report (and clear) any error a kernel recorded on
 * the device since the last check: KDA_ERR_TIMEOUT for an expired bounded
 * wait, KDA_ERR_SHAPE for cu_seqlens that break the rules of the varlen
 * entry points, KDA_ERR_CUDA for a runtime error. */
kda_status kda_check(void* stream);

/* Diagnostics: per-kernel device timing.  kda_timing_enable(1) clears the
 * totals and, until kda_timing_enable(0), brackets every kernel the library
 * launches with two CUDA events recorded on that launch's stream (the events
 * are created on first use and reused).  kda_timing_count() returns the
 * number of distinct kernel names seen; kda_timing_entry(i, ...) copies the
 * i-th name (NUL-terminated, truncated to name_len), its summed device time
 * in milliseconds and its launch count, and returns 0 (-1 if i is out of
 * range).  Both readers wait for the recorded events.  Not for use inside
 * CUDA graph capture. */
void kda_timing_enable(int on);
int kda_timing_count(void);
int kda_timing_entry(int i, char* name, int name_len, double* total_ms, long* launches);

/* Diagnostics: self-test of the tensor-core building blocks.  Computes
 * D[128 x N] = A[128 x 64] * B[N x 64]^T (D fp32 row-major; N = 64 or 128;
 * all device pointers) with one tcgen05 MMA chain from 128B-swizzled
 * shared-memory tiles.  flags: bit 0 stage by TMA (else by thread stores);
 * bit 1 A is given K-minor, i.e. as A^T [64][128] row-major (MN-major
 * operand, TMA only); bit 2 B likewise as B^T [64][N].  Other bits are
 * rejected with KDA_ERR_INVALID_ARG.  *status (device int, caller-zeroed) is
 * set to 1 if a bounded device wait expired. */
kda_status kda_selftest_mma(const void* A, const void* B, float* D, int N, int flags,
                            int* status, void* stream);

/* Diagnostics: the bounded-wait error path of the tensor-core kernels.  One
 * warp waits, with a limit of limit_cycles (0 .. 4e9) SM clock cycles, on an
 * mbarrier that nothing arrives at, through the same wait routine the chunk
 * kernels use; it gives up, records the error and returns with nothing in
 * flight.  The next kda_check on the stream then returns KDA_ERR_TIMEOUT
 * and clears it. */
kda_status kda_selftest_wait_timeout(long long limit_cycles, void* stream);

/* Static description of a status code. */
const char* kda_status_str(kda_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
