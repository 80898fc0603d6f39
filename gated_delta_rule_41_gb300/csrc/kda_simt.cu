// Generic fp32 CUDA-core (SIMT) chunk scan: any K, V <= 128, chunk 16/32/64
// or 128, f32 or bf16 inputs, all arithmetic in fp32.
//
// Chunk form (K3 README, table 实现路线表, row L2: (1) cumsum of the clamped
// gate inside each chunk, (2) the lower-triangular system, (3) the solve,
// (4) the state passed between chunks).  Per head and chunk of C rows, with
// qs = scale*q, G_r = sum_{s<=r} max(g_s,-5) and gl = G_{C-1}:
//     A[i][j]   = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)      j < i
//     T         = (I + A)^{-1}
//     W         = T diag(beta) (k o exp(G)),  U = T diag(beta) v
//     Aqk[r][j] = sum_c qs_rc k_jc exp(G_rc - G_jc)            j <= r
//     Qh = qs o exp(G),  Kb = k o exp(gl - G),  gam = exp(gl)
//     delta = U - W S;  O = Qh S + Aqk delta;  S <- diag(gam) S + Kb^T delta
// Backward of those steps, chunk by chunk in reverse, with dS the gradient of
// the state at the END of the chunk and S0 the state at its start:
//     ddelta = Aqk^T dO + Kb dS
//     dS0    = diag(gam) dS + Qh^T dO - W^T ddelta
//     dQh = dO S0^T, dW = -ddelta S0^T, dKb = delta dS^T, dgam = rowsum(dS o S0)
//     dAqk = mask(dO delta^T), dU = ddelta
//     dT = mask_strict(dU (beta v)^T + dW (beta k o exp(G))^T)
//     dA = -mask_strict(T^T dT T^T);   d(beta v) = T^T dU;  d(beta khat) = T^T dW
// then through the pairwise decays into dq, dk, dbeta, dG, and
// dg_s = [g_s >= -5] * sum_{r>=s} dG_r.
//
// Kernels (one launch each, all stream ordered):
//   intra   (chunk, head)    : G, A, T, Aqk, W, U, Qh, Kb, gam     -> workspace
//   state_f (V tile, head)   : sequential over chunks; delta, o, h, ht
//   state_b (V tile, head)   : reverse over chunks; dh (= dS), ddelta, dh0
//   vgrad   (chunk, head)    : contractions over V (dQh, dW, dKb, dgam, dAqk,
//                              dTv, dv, dbeta from v)
//   kgrad   (chunk, head)    : chunk-local algebra over C and K -> dq, dk, dg, dbeta
//   group   (token)          : GVA sum of dq, dk over value heads, cast
#include <algorithm>

#include "kda_common.cuh"
#include "kda_timing.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kVT = 32;  // value columns per CTA in the state passes
// Chunks of 128 rows (BIG instantiations): a chunk's C x C matrices and
// some C x K arrays no longer fit in shared memory beside its k, q and G
// rows, so they live in a per-(chunk, head) scratch area of the workspace
// (5 C (C + 1) floats), the state passes read their operands from the
// workspace arrays directly, and the per-thread result arrays hold
// C * max(C, K) / 256 = 64 values.
constexpr int kScratchMats = 5;

struct Ws {
    float *W, *U, *Qh, *Kb, *Aqk, *Tm, *gam, *dlt;   // forward quantities
    float *hs, *dhs, *ddl;                           // bwd: states, state grads, ddelta
    float *dQh, *dWm, *dKb, *dgam, *dAqk, *dTv, *dbv;  // bwd: V contractions
    float *dqh, *dkh;                                // bwd: dq, dk per value head (fp32)
    float* scr;   // C > 64: kScratchMats C x (C + 1) floats per (chunk, head)
};

struct Dims {
    int B, T, H, HV, K, V, C, NT, G;
    float scale;
    int qkn;   // L2-normalise q and k over K inside the kernels
    // Variable-length sequences (B == 1, sequences packed along T): ctab
    // [NT][2] holds each chunk's first token and number of valid rows (0 for
    // an unused slot), sfirst [nseq + 1] each sequence's first chunk.  T is
    // then NT * C (the workspace's padded length) and Tr the real token
    // count.  ctab == nullptr: fixed-length batches, Tr == T.
    int Tr;
    const int* ctab;
    const int* sfirst;
    int NS;   // rows of the state arrays: B * HV, or nseq * HV with a chunk table
};

// Chunk n of head row bh: batch b, first token t0 and valid rows len (len <
// C only for the last chunk of a variable-length sequence; 0 for an unused
// chunk-table slot).  With a chunk table the head row is hv (B == 1).
struct ChunkRef {
    int b, t0, len;
};
__device__ __forceinline__ ChunkRef chunk_ref(const Dims& d, int bh, int n) {
    if (!d.ctab) return ChunkRef{bh / d.HV, n * d.C, d.C};
    return ChunkRef{0, d.ctab[2 * n], d.ctab[2 * n + 1]};
}

Dims make_dims(const kda_dims& d) {
    Dims r;
    r.B = d.B; r.T = d.T; r.H = d.H; r.HV = d.HV; r.K = d.K; r.V = d.V;
    r.C = d.chunk_size; r.NT = d.T / d.chunk_size; r.G = d.HV / d.H; r.scale = d.scale;
    r.qkn = d.qk_l2norm != 0;
    r.Tr = d.T;
    r.ctab = nullptr;
    r.sfirst = nullptr;
    r.NS = d.B * d.HV;
    return r;
}

// Workspace carve-up; returns the total size.  With base == nullptr only sizes.
size_t carve(const Dims& d, int for_bwd, char* base, Ws* w) {
    const size_t BH = (size_t)d.B * d.HV, T = d.T, K = d.K, V = d.V, C = d.C, NT = d.NT;
    size_t off = 0;
    auto take = [&](size_t nfloats) {
        float* p = base ? reinterpret_cast<float*>(base + off) : nullptr;
        off += align256(nfloats * sizeof(float));
        return p;
    };
    Ws x{};
    x.W = take(BH * T * K);
    x.U = take(BH * T * V);
    x.Qh = take(BH * T * K);
    x.Kb = take(BH * T * K);
    x.Aqk = take(BH * NT * C * C);
    x.Tm = take(BH * NT * C * C);
    x.gam = take(BH * NT * K);
    x.dlt = take(BH * T * V);
    if (C > 64) x.scr = take(BH * NT * kScratchMats * C * (C + 1));
    if (for_bwd) {
        x.hs = take(BH * NT * K * V);
        x.dhs = take(BH * NT * K * V);
        x.ddl = take(BH * T * V);
        x.dQh = take(BH * T * K);
        x.dWm = take(BH * T * K);
        x.dKb = take(BH * T * K);
        x.dgam = take(BH * NT * K);
        x.dAqk = take(BH * NT * C * C);
        x.dTv = take(BH * NT * C * C);
        x.dbv = take(BH * T);
        x.dqh = take((size_t)d.B * T * d.HV * K);
        x.dkh = take((size_t)d.B * T * d.HV * K);
    }
    if (w) *w = x;
    return off;
}

__device__ __forceinline__ size_t tok_idx(const Dims& d, int b, int t, int head, int nheads,
                                          int width) {
    return (((size_t)b * d.T + t) * nheads + head) * width;
}

// L2 normalisation of q and k rows in place: kS holds k, qS holds scale * q
// (C rows of K floats, row stride KP).  Afterwards kS holds k / max(|k|, eps)
// and qS holds scale * q / max(|q|, eps).  One warp per row.
constexpr float kNormEps = 1e-12f;

__device__ __forceinline__ void l2norm_rows(float* kS, float* qS, int C, int K, int KP,
                                            float scale) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < C; r += kThreads / 32) {
        float sk = 0.f, sq = 0.f;
        for (int c = lane; c < K; c += 32) {
            const float kv = kS[r * KP + c], qv = qS[r * KP + c];
            sk = fmaf(kv, kv, sk);
            sq = fmaf(qv, qv, sq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
        }
        // |q| = |scale q| / scale
        const float ik = 1.f / fmaxf(sqrtf(sk), kNormEps);
        const float iq = 1.f / fmaxf(sqrtf(sq) / scale, kNormEps);
        for (int c = lane; c < K; c += 32) {
            kS[r * KP + c] *= ik;
            qS[r * KP + c] *= iq;
        }
    }
}

// ---------------------------------------------------------------------------
// intra: per (chunk, head)
// smem: k[C][K+1], qs[C][K+1], G[C][K+1], A[C][C+1], Tm[C][C+1], beta[C]
// ---------------------------------------------------------------------------
// (BIG: A and Tm in the chunk's scratch area instead)
size_t intra_smem(const Dims& d) {
    const size_t mats = d.C > 64 ? 0 : 2 * (size_t)d.C * (d.C + 1);
    return sizeof(float) * (3 * (size_t)d.C * (d.K + 1) + mats + d.C);
}

template <typename Tin, bool BIG>
__global__ void __launch_bounds__(kThreads)
intra_kernel(Dims d, Ws w, const Tin* __restrict__ q, const Tin* __restrict__ k,
             const Tin* __restrict__ v, const Tin* __restrict__ g, const Tin* __restrict__ beta) {
    const int n = blockIdx.x, bh = blockIdx.y;
    const ChunkRef cr = chunk_ref(d, bh, n);
    if (cr.len <= 0) return;
    const int b = cr.b, hv = bh % d.HV, h = hv / d.G;
    const int C = d.C, K = d.K, V = d.V, KP = K + 1, CP = C + 1;
    const int tid = threadIdx.x;
    extern __shared__ float sm[];
    float* kS = sm;
    float* qS = kS + C * KP;
    float* GS = qS + C * KP;
    float* A = BIG ? w.scr + ((size_t)bh * d.NT + n) * kScratchMats * C * CP : GS + C * KP;
    float* Tm = A + C * CP;
    float* bS = BIG ? GS + C * KP : Tm + C * CP;
    const int t0 = cr.t0, len = cr.len;

    // rows past a sequence's end enter as q = k = v = 0, g = 0, beta = 0:
    // they leave the state unchanged and their outputs are not written
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        const bool on = r < len;
        const size_t iq = tok_idx(d, b, t0 + r, h, d.H, K) + c;
        const size_t ig = tok_idx(d, b, t0 + r, hv, d.HV, K) + c;
        kS[r * KP + c] = on ? to_f(k[iq]) : 0.f;
        qS[r * KP + c] = on ? d.scale * to_f(q[iq]) : 0.f;
        GS[r * KP + c] = on ? fmaxf(to_f(g[ig]), kGateFloor) : 0.f;
    }
    for (int r = tid; r < C; r += kThreads)
        bS[r] = r < len ? to_f(beta[((size_t)b * d.T + t0 + r) * d.HV + hv]) : 0.f;
    __syncthreads();
    if (d.qkn) {
        l2norm_rows(kS, qS, C, K, KP, d.scale);
        __syncthreads();
    }
    for (int c = tid; c < K; c += kThreads) {  // (1) in-chunk cumsum
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += GS[r * KP + c];
            GS[r * KP + c] = acc;
        }
    }
    __syncthreads();

    // (2) A (strictly lower, beta-scaled) and Aqk (lower incl. diagonal)
    float* Aqk_g = w.Aqk + ((size_t)bh * d.NT + n) * C * C;
    for (int p = tid; p < C * C; p += kThreads) {
        const int i = p % C, j = p / C;
        float a = 0.f, aq = 0.f;
        if (j <= i) {
            for (int c = 0; c < K; ++c) {
                const float e = expf(GS[i * KP + c] - GS[j * KP + c]);
                const float kj = kS[j * KP + c] * e;
                a += kS[i * KP + c] * kj;
                aq += qS[i * KP + c] * kj;
            }
        }
        A[i * CP + j] = j < i ? bS[i] * a : 0.f;
        Aqk_g[i * C + j] = j <= i ? aq : 0.f;
    }
    __syncthreads();

    // (3) T = (I + A)^{-1}; column j solved top to bottom
    for (int j = tid; j < C; j += kThreads) {
        for (int i = 0; i < j; ++i) Tm[i * CP + j] = 0.f;
        Tm[j * CP + j] = 1.f;
        for (int i = j + 1; i < C; ++i) {
            float acc = 0.f;
            for (int m = j; m < i; ++m) acc += A[i * CP + m] * Tm[m * CP + j];
            Tm[i * CP + j] = -acc;
        }
    }
    __syncthreads();

    float* Tm_g = w.Tm + ((size_t)bh * d.NT + n) * C * C;
    for (int p = tid; p < C * C; p += kThreads) Tm_g[p] = Tm[(p / C) * CP + p % C];
    const size_t row0 = (size_t)bh * d.T + (size_t)n * C;
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        const float G = GS[r * KP + c], gl = GS[(C - 1) * KP + c];
        w.Qh[(row0 + r) * K + c] = qS[r * KP + c] * expf(G);
        w.Kb[(row0 + r) * K + c] = kS[r * KP + c] * expf(gl - G);
        kS[r * KP + c] = bS[r] * kS[r * KP + c] * expf(G);  // beta k o exp(G), in place
    }
    for (int c = tid; c < K; c += kThreads)
        w.gam[((size_t)bh * d.NT + n) * K + c] = expf(GS[(C - 1) * KP + c]);
    __syncthreads();

    // W = T (beta k o exp(G)),  U = T (beta v)
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        float acc = 0.f;
        for (int m = 0; m <= r; ++m) acc += Tm[r * CP + m] * kS[m * KP + c];
        w.W[(row0 + r) * K + c] = acc;
    }
    for (int i = tid; i < C * V; i += kThreads) {
        const int r = i / V, j = i % V;
        float acc = 0.f;
        for (int m = 0; m <= r && m < len; ++m)
            acc += Tm[r * CP + m] * bS[m] * to_f(v[tok_idx(d, b, t0 + m, hv, d.HV, V) + j]);
        w.U[(row0 + r) * V + j] = acc;
    }
}

// ---------------------------------------------------------------------------
// state_f: per (V tile of kVT columns, head); sequential over chunks.
// mode bits: 1 = write o, 2 = store h (state at chunk start) and delta.
// smem: W[C][K], Qh[C][K], Kb[C][K], Aqk[C][C], gam[K], S[K][VT], U/delta[C][VT]
// ---------------------------------------------------------------------------
// (BIG: W, Qh, Kb and Aqk are read from the workspace arrays in place)
size_t statef_smem(const Dims& d) {
    const size_t ops = d.C > 64 ? 0 : 3 * (size_t)d.C * d.K + (size_t)d.C * d.C;
    return sizeof(float) * (ops + d.K + (size_t)d.K * kVT + 2 * (size_t)d.C * kVT);
}

template <typename Tout, bool BIG>
__global__ void __launch_bounds__(kThreads)
state_fwd_kernel(Dims d, Ws w, const float* __restrict__ h0, Tout* __restrict__ o,
                 float* __restrict__ ht, int mode) {
    // bh: the state's row (b, hv), or (sequence, hv) with a chunk table;
    // bw: the head row of the workspace arrays
    const int vt = blockIdx.x, bh = blockIdx.y;
    const int hv = bh % d.HV, bw = d.ctab ? hv : bh;
    const int nfirst = d.ctab ? d.sfirst[bh / d.HV] : 0;
    const int nend = d.ctab ? d.sfirst[bh / d.HV + 1] : d.NT;
    const int C = d.C, K = d.K, V = d.V;
    const int j0 = vt * kVT;
    const int VT = min(kVT, V - j0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ float sm[];
    const int ops = BIG ? 0 : 3 * C * K + C * C;
    float* Ws_ = sm;
    float* Qs = Ws_ + C * K;
    float* Kbs = Qs + C * K;
    float* As = Kbs + C * K;
    float* gs = sm + ops;
    float* S = gs + K;
    float* Us = S + K * kVT;
    float* Ds = Us + C * kVT;

    for (int i = tid; i < K * kVT; i += kThreads) {
        const int c = i / kVT, j = i % kVT;
        S[i] = (h0 && j < VT) ? h0[((size_t)bh * K + c) * V + j0 + j] : 0.f;
    }
    for (int n = nfirst; n < nend; ++n) {
        __syncthreads();
        const ChunkRef cr = chunk_ref(d, bw, n);
        const size_t row0 = (size_t)bw * d.T + (size_t)n * C;
        if (BIG) {
            Ws_ = w.W + row0 * K;
            Qs = w.Qh + row0 * K;
            Kbs = w.Kb + row0 * K;
            As = w.Aqk + ((size_t)bw * d.NT + n) * C * C;
        } else {
            for (int i = tid; i < C * K; i += kThreads) {
                Ws_[i] = w.W[row0 * K + i];
                Qs[i] = w.Qh[row0 * K + i];
                Kbs[i] = w.Kb[row0 * K + i];
            }
            for (int i = tid; i < C * C; i += kThreads)
                As[i] = w.Aqk[((size_t)bw * d.NT + n) * C * C + i];
        }
        for (int c = tid; c < K; c += kThreads) gs[c] = w.gam[((size_t)bw * d.NT + n) * K + c];
        for (int i = tid; i < C * kVT; i += kThreads) {
            const int r = i / kVT, j = i % kVT;
            Us[i] = j < VT ? w.U[(row0 + r) * V + j0 + j] : 0.f;
        }
        if (mode & 2) {
            float* hs = w.hs + ((size_t)bw * d.NT + n) * K * V;
            for (int i = tid; i < K * kVT; i += kThreads) {
                const int c = i / kVT, j = i % kVT;
                if (j < VT) hs[(size_t)c * V + j0 + j] = S[i];
            }
        }
        __syncthreads();
        // delta = U - W S   (thread: column lane, rows warp + 8i)
        for (int r = warp; r < C; r += kThreads / 32) {
            float acc = 0.f;
            for (int c = 0; c < K; ++c) acc += Ws_[r * K + c] * S[c * kVT + lane];
            const float dl = Us[r * kVT + lane] - acc;
            Ds[r * kVT + lane] = dl;
            if ((mode & 2) && lane < VT) w.dlt[(row0 + r) * V + j0 + lane] = dl;
        }
        __syncthreads();
        if (mode & 1) {  // O = Qh S + Aqk delta
            for (int r = warp; r < C; r += kThreads / 32) {
                float acc = 0.f;
                for (int c = 0; c < K; ++c) acc += Qs[r * K + c] * S[c * kVT + lane];
                for (int m = 0; m <= r; ++m) acc += As[r * C + m] * Ds[m * kVT + lane];
                if (lane < VT && r < cr.len)
                    o[tok_idx(d, cr.b, cr.t0 + r, hv, d.HV, V) + j0 + lane] = from_f<Tout>(acc);
            }
        }
        __syncthreads();
        // S <- diag(gam) S + Kb^T delta
        for (int c = warp; c < K; c += kThreads / 32) {
            float acc = gs[c] * S[c * kVT + lane];
            for (int m = 0; m < C; ++m) acc += Kbs[m * K + c] * Ds[m * kVT + lane];
            S[c * kVT + lane] = acc;
        }
    }
    __syncthreads();
    if (ht) {
        for (int i = tid; i < K * kVT; i += kThreads) {
            const int c = i / kVT, j = i % kVT;
            if (j < VT) ht[((size_t)bh * K + c) * V + j0 + j] = S[i];
        }
    }
}

// ---------------------------------------------------------------------------
// state_b: per (V tile, head); reverse over chunks.
// smem: W[C][K], Qh[C][K], Kb[C][K], Aqk[C][C], gam[K], dS[K][VT], dO[C][VT], dd[C][VT]
// ---------------------------------------------------------------------------
template <typename Tin, bool BIG>
__global__ void __launch_bounds__(kThreads)
state_bwd_kernel(Dims d, Ws w, const Tin* __restrict__ dout, const float* __restrict__ dht,
                 float* __restrict__ dh0) {
    const int vt = blockIdx.x, bh = blockIdx.y;
    const int hv = bh % d.HV, bw = d.ctab ? hv : bh;
    const int nfirst = d.ctab ? d.sfirst[bh / d.HV] : 0;
    const int nend = d.ctab ? d.sfirst[bh / d.HV + 1] : d.NT;
    const int C = d.C, K = d.K, V = d.V;
    const int j0 = vt * kVT;
    const int VT = min(kVT, V - j0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ float sm[];
    const int ops = BIG ? 0 : 3 * C * K + C * C;
    float* Ws_ = sm;
    float* Qs = Ws_ + C * K;
    float* Kbs = Qs + C * K;
    float* As = Kbs + C * K;
    float* gs = sm + ops;
    float* dS = gs + K;
    float* dOs = dS + K * kVT;
    float* dds = dOs + C * kVT;

    for (int i = tid; i < K * kVT; i += kThreads) {
        const int c = i / kVT, j = i % kVT;
        dS[i] = (dht && j < VT) ? dht[((size_t)bh * K + c) * V + j0 + j] : 0.f;
    }
    for (int n = nend - 1; n >= nfirst; --n) {
        __syncthreads();
        const ChunkRef cr = chunk_ref(d, bw, n);
        const size_t row0 = (size_t)bw * d.T + (size_t)n * C;
        if (BIG) {
            Ws_ = w.W + row0 * K;
            Qs = w.Qh + row0 * K;
            Kbs = w.Kb + row0 * K;
            As = w.Aqk + ((size_t)bw * d.NT + n) * C * C;
        } else {
            for (int i = tid; i < C * K; i += kThreads) {
                Ws_[i] = w.W[row0 * K + i];
                Qs[i] = w.Qh[row0 * K + i];
                Kbs[i] = w.Kb[row0 * K + i];
            }
            for (int i = tid; i < C * C; i += kThreads)
                As[i] = w.Aqk[((size_t)bw * d.NT + n) * C * C + i];
        }
        for (int c = tid; c < K; c += kThreads) gs[c] = w.gam[((size_t)bw * d.NT + n) * K + c];
        for (int i = tid; i < C * kVT; i += kThreads) {
            const int r = i / kVT, j = i % kVT;
            dOs[i] = (j < VT && r < cr.len)
                         ? to_f(dout[tok_idx(d, cr.b, cr.t0 + r, hv, d.HV, V) + j0 + j])
                         : 0.f;
        }
        {
            float* dh = w.dhs + ((size_t)bw * d.NT + n) * K * V;
            for (int i = tid; i < K * kVT; i += kThreads) {
                const int c = i / kVT, j = i % kVT;
                if (j < VT) dh[(size_t)c * V + j0 + j] = dS[i];
            }
        }
        __syncthreads();
        // ddelta = Aqk^T dO + Kb dS
        for (int r = warp; r < C; r += kThreads / 32) {
            float acc = 0.f;
            for (int t = r; t < C; ++t) acc += As[t * C + r] * dOs[t * kVT + lane];
            for (int c = 0; c < K; ++c) acc += Kbs[r * K + c] * dS[c * kVT + lane];
            dds[r * kVT + lane] = acc;
            if (lane < VT) w.ddl[(row0 + r) * V + j0 + lane] = acc;
        }
        __syncthreads();
        // dS0 = diag(gam) dS + Qh^T dO - W^T ddelta
        for (int c = warp; c < K; c += kThreads / 32) {
            float acc = gs[c] * dS[c * kVT + lane];
            for (int r = 0; r < C; ++r)
                acc += Qs[r * K + c] * dOs[r * kVT + lane] - Ws_[r * K + c] * dds[r * kVT + lane];
            dS[c * kVT + lane] = acc;
        }
    }
    __syncthreads();
    if (dh0) {
        for (int i = tid; i < K * kVT; i += kThreads) {
            const int c = i / kVT, j = i % kVT;
            if (j < VT) dh0[((size_t)bh * K + c) * V + j0 + j] = dS[i];
        }
    }
}

// ---------------------------------------------------------------------------
// vgrad: per (chunk, head); contractions over V, in slices of 32 columns.
// smem: S0[K][33], dS[K][33], dl[C][33], dd[C][33], dO[C][33], v[C][33],
//       Tm[C][C+1], beta[C], dbv[C]
// ---------------------------------------------------------------------------
constexpr int kVS = 32, kVSP = 33;
constexpr int kMaxPer = 32;  // C*K/256 and C*C/256 upper bounds (C<=64, K<=128)
constexpr int kMaxPerBig = 64;  // the same for C = 128

size_t vgrad_smem(const Dims& d) {
    return sizeof(float) * (2 * (size_t)d.K * kVSP + 4 * (size_t)d.C * kVSP +
                            (size_t)d.C * (d.C + 1) + 2 * (size_t)d.C);
}

template <typename Tin, bool BIG>
__global__ void __launch_bounds__(kThreads)
vgrad_kernel(Dims d, Ws w, const Tin* __restrict__ v, const Tin* __restrict__ beta,
             const Tin* __restrict__ dout, Tin* __restrict__ dv) {
    const int n = blockIdx.x, bh = blockIdx.y;
    const ChunkRef cr = chunk_ref(d, bh, n);
    if (cr.len <= 0) return;
    const int b = cr.b, hv = bh % d.HV, t0 = cr.t0, len = cr.len;
    const int C = d.C, K = d.K, V = d.V, CP = C + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int KMP = BIG ? kMaxPerBig : kMaxPer;
    constexpr int UNR = BIG ? 1 : KMP;   // (BIG: the arrays live in local memory)
    extern __shared__ float sm[];
    float* S0 = sm;
    float* dSs = S0 + K * kVSP;
    float* dls = dSs + K * kVSP;
    float* dds = dls + C * kVSP;
    float* dOs = dds + C * kVSP;
    float* vs = dOs + C * kVSP;
    float* Tm = vs + C * kVSP;
    float* bS = Tm + C * CP;
    float* dbv = bS + C;

    const size_t row0 = (size_t)bh * d.T + (size_t)n * C;
    const float* hs = w.hs + ((size_t)bh * d.NT + n) * K * V;
    const float* dh = w.dhs + ((size_t)bh * d.NT + n) * K * V;
    for (int p = tid; p < C * C; p += kThreads) Tm[(p / C) * CP + p % C] = w.Tm[((size_t)bh * d.NT + n) * C * C + p];
    for (int r = tid; r < C; r += kThreads) {
        bS[r] = r < len ? to_f(beta[((size_t)b * d.T + t0 + r) * d.HV + hv]) : 0.f;
        dbv[r] = 0.f;
    }

    // ownership: (r, c) outputs with c = tid % K, r = tid / K + i * (256 / K)
    const int ck = tid % K, rstep = kThreads / K;
    const int nrk = (C * K + kThreads - 1) / kThreads;
    // (r, m) outputs with m = tid % C, r = tid / C + i * (256 / C)
    const int mc = tid % C, rcstep = kThreads / C;
    const int nrc = (C * C + kThreads - 1) / kThreads;
    float aQ[KMP], aW[KMP], aKb[KMP], aAq[KMP], aTv[KMP];
#pragma unroll UNR
    for (int i = 0; i < KMP; ++i) aQ[i] = aW[i] = aKb[i] = aAq[i] = aTv[i] = 0.f;
    float agam = 0.f;

    for (int j0 = 0; j0 < V; j0 += kVS) {
        const int VS = min(kVS, V - j0);
        __syncthreads();
        for (int i = tid; i < K * kVS; i += kThreads) {
            const int c = i / kVS, j = i % kVS;
            const bool ok = j < VS;
            S0[c * kVSP + j] = ok ? hs[(size_t)c * V + j0 + j] : 0.f;
            dSs[c * kVSP + j] = ok ? dh[(size_t)c * V + j0 + j] : 0.f;
        }
        for (int i = tid; i < C * kVS; i += kThreads) {
            const int r = i / kVS, j = i % kVS;
            const bool ok = j < VS;
            dls[r * kVSP + j] = ok ? w.dlt[(row0 + r) * V + j0 + j] : 0.f;
            dds[r * kVSP + j] = ok ? w.ddl[(row0 + r) * V + j0 + j] : 0.f;
            const size_t it = tok_idx(d, b, t0 + r, hv, d.HV, V) + j0 + j;
            dOs[r * kVSP + j] = ok && r < len ? to_f(dout[it]) : 0.f;
            vs[r * kVSP + j] = ok && r < len ? to_f(v[it]) : 0.f;
        }
        __syncthreads();
        // C x K contractions
        for (int j = 0; j < kVS; ++j) {
            const float s0 = S0[ck * kVSP + j], ds = dSs[ck * kVSP + j];
            if (tid < K) agam += ds * s0;
#pragma unroll UNR
            for (int i = 0; i < KMP; ++i) {
                if (i < nrk) {
                    const int r = tid / K + i * rstep;
                    if (r < C) {
                        aQ[i] += dOs[r * kVSP + j] * s0;
                        aW[i] -= dds[r * kVSP + j] * s0;
                        aKb[i] += dls[r * kVSP + j] * ds;
                    }
                }
            }
        }
        // C x C contractions
        for (int j = 0; j < kVS; ++j) {
            const float dlm = dls[mc * kVSP + j], vm = vs[mc * kVSP + j];
#pragma unroll UNR
            for (int i = 0; i < KMP; ++i) {
                if (i < nrc) {
                    const int r = tid / C + i * rcstep;
                    if (r < C) {
                        aAq[i] += dOs[r * kVSP + j] * dlm;
                        aTv[i] += dds[r * kVSP + j] * vm;
                    }
                }
            }
        }
        // d(beta v) = T^T ddelta -> dv = beta * that; dbeta += sum_j that * v
        for (int m = warp; m < C; m += kThreads / 32) {
            float acc = 0.f;
            for (int i = m; i < C; ++i) acc += Tm[i * CP + m] * dds[i * kVSP + lane];
            if (lane < VS && m < len)
                dv[tok_idx(d, b, t0 + m, hv, d.HV, V) + j0 + lane] = from_f<Tin>(bS[m] * acc);
            float pb = lane < VS ? acc * vs[m * kVSP + lane] : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) pb += __shfl_xor_sync(0xffffffffu, pb, off);
            if (lane == 0) dbv[m] += pb;
        }
    }
    __syncthreads();
#pragma unroll UNR
    for (int i = 0; i < KMP; ++i) {
        if (i < nrk) {
            const int r = tid / K + i * rstep;
            if (r < C) {
                w.dQh[(row0 + r) * K + ck] = aQ[i];
                w.dWm[(row0 + r) * K + ck] = aW[i];
                w.dKb[(row0 + r) * K + ck] = aKb[i];
            }
        }
        if (i < nrc) {
            const int r = tid / C + i * rcstep;
            if (r < C) {
                const size_t base = ((size_t)bh * d.NT + n) * C * C;
                w.dAqk[base + r * C + mc] = mc <= r ? aAq[i] : 0.f;
                w.dTv[base + r * C + mc] = mc < r ? aTv[i] : 0.f;
            }
        }
    }
    if (tid < K) w.dgam[((size_t)bh * d.NT + n) * K + tid] = agam;
    for (int r = tid; r < C; r += kThreads) w.dbv[row0 + r] = dbv[r];
}

// ---------------------------------------------------------------------------
// kgrad: per (chunk, head); chunk-local algebra over C and K.
// smem: k[C][K+1], qs[C][K+1], G[C][K+1], X[C][K+1], Y[C][K+1],
//       Tm[C][C+1], dAqk[C][C+1], D[C][C+1], beta[C], dbeta[C]
// ---------------------------------------------------------------------------
// Factor tables for NB = C / 16 row blocks: Fb holds NB (NB + 1) / 2 block
// pairs, eGbS and eLbS NB blocks, each K wide.  (BIG: X, Y, Tm, dAqk and D
// in the chunk's scratch area instead of shared memory.)
size_t kgrad_smem(const Dims& d) {
    const size_t NB = d.C / 16;
    const size_t mats =
        d.C > 64 ? 0 : 2 * (size_t)d.C * (d.K + 1) + 3 * (size_t)d.C * (d.C + 1);
    return sizeof(float) * (3 * (size_t)d.C * (d.K + 1) + mats + 2 * d.C +
                            (NB * (NB + 1) / 2 + 2 * NB) * (size_t)d.K);
}

template <typename Tin, bool BIG>
__global__ void __launch_bounds__(kThreads)
kgrad_kernel(Dims d, Ws w, const Tin* __restrict__ q, const Tin* __restrict__ k,
             const Tin* __restrict__ g, const Tin* __restrict__ beta, Tin* __restrict__ dg,
             Tin* __restrict__ dbeta) {
    const int n = blockIdx.x, bh = blockIdx.y;
    const ChunkRef cr = chunk_ref(d, bh, n);
    if (cr.len <= 0) return;
    const int b = cr.b, hv = bh % d.HV, h = hv / d.G, len = cr.len;
    const int C = d.C, K = d.K, KP = K + 1, CP = C + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int KMP = BIG ? kMaxPerBig : kMaxPer;
    constexpr int UNR = BIG ? 1 : KMP;   // (BIG: the arrays live in local memory)
    const int NB = C / 16;
    extern __shared__ float sm[];
    float* kS = sm;
    float* qS = kS + C * KP;
    float* GS = qS + C * KP;
    // the five matrices: in shared memory, or (BIG) in the chunk's scratch
    // area, each C x (C + 1) floats there
    float* mats = BIG ? w.scr + ((size_t)bh * d.NT + n) * kScratchMats * C * CP : GS + C * KP;
    const int XS = BIG ? C * CP : C * KP;   // space of X and of Y
    float* X = mats;          // dW, then d(beta khat)
    float* Y = X + XS;        // beta khat, then dG
    float* Tm = Y + XS;
    float* dAq = Tm + C * CP;
    float* D = dAq + C * CP;  // dT -> dT T^T -> dA
    float* bS = BIG ? GS + C * KP : D + C * CP;
    float* dbS = bS + C;
    float* Fb = dbS + C;                    // Fb[fidx(R,J)*K + c] = exp(G_bR - G_bJ), J <= R
    float* eGbS = Fb + NB * (NB + 1) / 2 * K;   // eGbS[R*K + c] = exp(G_bR)
    float* eLbS = eGbS + NB * K;                // eLbS[R*K + c] = exp(G_last - G_bR)
    const int t0 = cr.t0;
    const size_t row0 = (size_t)bh * d.T + (size_t)n * C;
    const size_t cc0 = ((size_t)bh * d.NT + n) * C * C;

    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        const bool on = r < len;
        const size_t iq = tok_idx(d, b, t0 + r, h, d.H, K) + c;
        kS[r * KP + c] = on ? to_f(k[iq]) : 0.f;
        qS[r * KP + c] = on ? d.scale * to_f(q[iq]) : 0.f;
        GS[r * KP + c] =
            on ? fmaxf(to_f(g[tok_idx(d, b, t0 + r, hv, d.HV, K) + c]), kGateFloor) : 0.f;
        X[r * KP + c] = w.dWm[(row0 + r) * K + c];
    }
    for (int p = tid; p < C * C; p += kThreads) {
        Tm[(p / C) * CP + p % C] = w.Tm[cc0 + p];
        dAq[(p / C) * CP + p % C] = w.dAqk[cc0 + p];
    }
    for (int r = tid; r < C; r += kThreads) {
        bS[r] = r < len ? to_f(beta[((size_t)b * d.T + t0 + r) * d.HV + hv]) : 0.f;
        dbS[r] = w.dbv[row0 + r];
    }
    __syncthreads();
    if (d.qkn) {
        l2norm_rows(kS, qS, C, K, KP, d.scale);
        __syncthreads();
    }
    for (int c = tid; c < K; c += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += GS[r * KP + c];
            GS[r * KP + c] = acc;
        }
    }
    __syncthreads();
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        Y[r * KP + c] = bS[r] * kS[r * KP + c] * expf(GS[r * KP + c]);
    }
    __syncthreads();
    // dT[i][m] = beta_m dTv[i][m] + sum_c dW[i][c] (beta khat)[m][c], m < i
    for (int p = tid; p < C * C; p += kThreads) {
        const int m = p % C, i = p / C;
        float acc = 0.f;
        if (m < i) {
            acc = bS[m] * w.dTv[cc0 + i * C + m];
            for (int c = 0; c < K; ++c) acc += X[i * KP + c] * Y[m * KP + c];
        }
        D[i * CP + m] = acc;
    }
    __syncthreads();
    // dbeta += sum_c d(beta khat)[m][c] khat[m][c], with d(beta khat) = T^T dW
    // and in the same pass: X <- T^T dW
    {
        float reg[KMP];
        const int nr = (C * K + kThreads - 1) / kThreads;
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            reg[u] = 0.f;
            if (u < nr) {
                const int i = tid + u * kThreads;
                if (i < C * K) {
                    const int m = i / K, c = i % K;
                    float acc = 0.f;
                    for (int r = m; r < C; ++r) acc += Tm[r * CP + m] * X[r * KP + c];
                    reg[u] = acc;
                }
            }
        }
        __syncthreads();
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            if (u < nr) {
                const int i = tid + u * kThreads;
                if (i < C * K) X[(i / K) * KP + i % K] = reg[u];
            }
        }
        // Y2 = dT T^T  (into registers, then back into D)
        const int nrc = (C * C + kThreads - 1) / kThreads;
        float rc[KMP];
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            rc[u] = 0.f;
            if (u < nrc) {
                const int p = tid + u * kThreads;
                if (p < C * C) {
                    const int i = p / C, j = p % C;
                    float acc = 0.f;
                    for (int m = 0; m < C; ++m) acc += D[i * CP + m] * Tm[j * CP + m];
                    rc[u] = acc;
                }
            }
        }
        __syncthreads();
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            if (u < nrc) {
                const int p = tid + u * kThreads;
                if (p < C * C) D[(p / C) * CP + p % C] = rc[u];
            }
        }
        __syncthreads();
        // dA = -mask_strict(T^T Y2)
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            rc[u] = 0.f;
            if (u < nrc) {
                const int p = tid + u * kThreads;
                if (p < C * C) {
                    const int i = p / C, j = p % C;
                    float acc = 0.f;
                    if (j < i)
                        for (int m = 0; m < C; ++m) acc += Tm[m * CP + i] * D[m * CP + j];
                    rc[u] = -acc;
                }
            }
        }
        __syncthreads();
#pragma unroll UNR
        for (int u = 0; u < KMP; ++u) {
            if (u < nrc) {
                const int p = tid + u * kThreads;
                if (p < C * C) D[(p / C) * CP + p % C] = rc[u];
            }
        }
    }
    __syncthreads();

    // Per element (r, c): direct terms and the pairwise-decay terms
    //   sA = sum_{j<r} dA[r][j] k_j e(r,j),   sQ = sum_{j<=r} dAqk[r][j] k_j e(r,j)
    //   cA = sum_{t>r} dA[t][r] beta_t k_t e(t,r),  cQ = sum_{t>=r} dAqk[t][r] qs_t e(t,r)
    // with e(t,j) = exp(G_t - G_j).  The decay is factored per 16-row block
    // (reference b = first row of the block): e(t,j) = E_t F[R(t)][R(j)] / E_j
    // with E_r = exp(G_r - G_b(r)) in [e^-75, 1] and F[R][J] = exp(G_bR - G_bJ),
    // so the inner loops are plain FMAs over tables and no factor overflows.
    auto fidx = [](int R, int J) { return R * (R + 1) / 2 + J; };
    for (int i = tid; i < NB * NB * K; i += kThreads) {
        const int R = i / (NB * K), J = (i / K) % NB, c = i % K;
        if (R < NB && J <= R)
            Fb[fidx(R, J) * K + c] = expf(GS[16 * R * KP + c] - GS[16 * J * KP + c]);
    }
    for (int i = tid; i < NB * K; i += kThreads) {
        const int R = i / K, c = i % K;
        eGbS[i] = expf(GS[16 * R * KP + c]);
        eLbS[i] = expf(GS[(C - 1) * KP + c] - GS[16 * R * KP + c]);
    }
    // Y <- KE[j][c] = k_j / E_j   (row-side table)
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        Y[r * KP + c] = kS[r * KP + c] * expf(GS[(r & ~15) * KP + c] - GS[r * KP + c]);
    }
    __syncthreads();
    const int nper = (C * K + kThreads - 1) / kThreads;
    float sAr[KMP], sQr[KMP], dKr[KMP];
#pragma unroll UNR
    for (int u = 0; u < KMP; ++u) {
        sAr[u] = sQr[u] = dKr[u] = 0.f;
        const int i = tid + u * kThreads;
        if (u < nper && i < C * K) {
            const int r = i / K, c = i % K, R = r >> 4;
            float sA = 0.f, sQ = 0.f;
            for (int J = 0; J <= R; ++J) {
                float pa = 0.f, pq = 0.f;
                const int jend = min(16 * J + 15, r);
                for (int j = 16 * J; j <= jend; ++j) {
                    const float ke = Y[j * KP + c];
                    pa += D[r * CP + j] * ke;  // D[r][r] = 0 (strictly lower)
                    pq += dAq[r * CP + j] * ke;
                }
                const float f = Fb[fidx(R, J) * K + c];
                sA += f * pa;
                sQ += f * pq;
            }
            const float E = expf(GS[r * KP + c] - GS[(r & ~15) * KP + c]);
            sAr[u] = sA * E;
            sQr[u] = sQ * E;
            dKr[u] = X[r * KP + c];  // d(beta khat)
        }
    }
    __syncthreads();
    // X <- KLb[t][c] = beta_t k_t E_t,  Y <- QL[t][c] = qs_t E_t   (column-side tables)
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        const float E = expf(GS[r * KP + c] - GS[(r & ~15) * KP + c]);
        X[r * KP + c] = bS[r] * kS[r * KP + c] * E;
        Y[r * KP + c] = qS[r * KP + c] * E;
    }
    __syncthreads();
    float dGr[KMP], dbr[KMP];
#pragma unroll UNR
    for (int u = 0; u < KMP; ++u) {
        dGr[u] = dbr[u] = 0.f;
        const int i = tid + u * kThreads;
        if (u < nper && i < C * K) {
            const int r = i / K, c = i % K, J = r >> 4;
            float cA = 0.f, cQ = 0.f;
            for (int R = J; R < NB; ++R) {
                float pa = 0.f, pq = 0.f;
                for (int t = max(16 * R, r); t < 16 * R + 16; ++t) {
                    pa += D[t * CP + r] * X[t * KP + c];  // D[r][r] = 0
                    pq += dAq[t * CP + r] * Y[t * KP + c];
                }
                const float f = Fb[fidx(R, J) * K + c];
                cA += f * pa;
                cQ += f * pq;
            }
            const float G = GS[r * KP + c];
            const float E = expf(G - GS[(r & ~15) * KP + c]);
            const float Einv = 1.f / E;
            cA *= Einv;
            cQ *= Einv;
            const float eG = eGbS[J * K + c] * E;      // exp(G_r)
            const float eL = eLbS[J * K + c] * Einv;   // exp(G_last - G_r)
            const float kr = kS[r * KP + c], qr = qS[r * KP + c];
            const float dKbeta = dKr[u], sA = sAr[u], sQ = sQr[u];
            const float dQh = w.dQh[(row0 + r) * K + c];
            const float dKb = w.dKb[(row0 + r) * K + c];
            const float br = bS[r];
            const float dk = br * dKbeta * eG + dKb * eL + br * sA + cA + cQ;
            const float dqs = dQh * eG + sQ;
            dGr[u] = dKbeta * br * kr * eG + dQh * qr * eG - dKb * kr * eL + br * kr * sA +
                     qr * sQ - kr * (cA + cQ);
            dbr[u] = dKbeta * kr * eG + kr * sA;
            if (r < len) {
                w.dqh[tok_idx(d, b, t0 + r, hv, d.HV, K) + c] = d.scale * dqs;
                w.dkh[tok_idx(d, b, t0 + r, hv, d.HV, K) + c] = dk;
            }
        }
    }
    __syncthreads();
#pragma unroll UNR
    for (int u = 0; u < KMP; ++u) {
        const int i = tid + u * kThreads;
        if (u < nper && i < C * K) {
            const int r = i / K, c = i % K;
            Y[r * KP + c] = dGr[u];
            X[r * KP + c] = dbr[u];
        }
    }
    __syncthreads();
    // last-row terms of dG: sum_r dKb_r Kb_r + dgam * gam
    for (int c = tid; c < K; c += kThreads) {
        const float gl = GS[(C - 1) * KP + c];
        float acc = w.dgam[((size_t)bh * d.NT + n) * K + c] * expf(gl);
        for (int r = 0; r < C; ++r)
            acc += w.dKb[(row0 + r) * K + c] * kS[r * KP + c] * expf(gl - GS[r * KP + c]);
        Y[(C - 1) * KP + c] += acc;
    }
    // dbeta per row
    for (int r = warp; r < C; r += kThreads / 32) {
        float acc = 0.f;
        for (int c = lane; c < K; c += 32) acc += X[r * KP + c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0 && r < len)
            dbeta[((size_t)b * d.T + t0 + r) * d.HV + hv] = from_f<Tin>(acc + dbS[r]);
    }
    __syncthreads();
    // dg_s = [g_s >= -5] sum_{r >= s} dG_r
    for (int c = tid; c < K; c += kThreads) {
        float acc = 0.f;
        for (int r = C - 1; r >= 0; --r) {
            acc += Y[r * KP + c];
            if (r < len) {
                const size_t ig = tok_idx(d, b, t0 + r, hv, d.HV, K) + c;
                dg[ig] = from_f<Tin>(to_f(g[ig]) >= kGateFloor ? acc : 0.f);
            }
        }
    }
}

// dq[b,t,h,:] = sum over the G value heads of the group (and the same for
// dk); with qkn, the sum is the gradient with respect to the normalised q
// (k), and the row is mapped back to the raw q (k):
//     dx = (dn - n <n, dn>) / max(|x|, eps),   n = x / max(|x|, eps).
// One warp per (b, t, h) row, K <= 128 (four channels per lane); cast to the dtype.
template <typename Tin>
__global__ void group_sum_kernel(Dims d, const float* __restrict__ dqh,
                                 const float* __restrict__ dkh, const Tin* __restrict__ q,
                                 const Tin* __restrict__ k, Tin* __restrict__ dq,
                                 Tin* __restrict__ dk) {
    const int lane = threadIdx.x & 31;
    const size_t rows = (size_t)d.B * d.Tr * d.H;
    const size_t wstep = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t row = blockIdx.x * (size_t)(blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += wstep) {
        const int h = row % d.H;
        const size_t bt = row / d.H;
        float sq[4], sk[4], xq[4], xk[4];
        float nq = 0.f, nk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = lane + 32 * e;
            sq[e] = sk[e] = xq[e] = xk[e] = 0.f;
            if (c < d.K) {
                for (int u = 0; u < d.G; ++u) {
                    const size_t j = (bt * d.HV + (size_t)h * d.G + u) * d.K + c;
                    sq[e] += dqh[j];
                    sk[e] += dkh[j];
                }
                if (d.qkn) {
                    xq[e] = to_f(q[row * d.K + c]);
                    xk[e] = to_f(k[row * d.K + c]);
                    nq = fmaf(xq[e], xq[e], nq);
                    nk = fmaf(xk[e], xk[e], nk);
                }
            }
        }
        if (d.qkn) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                nq += __shfl_xor_sync(0xffffffffu, nq, off);
                nk += __shfl_xor_sync(0xffffffffu, nk, off);
            }
            const float iq = 1.f / fmaxf(sqrtf(nq), kNormEps);
            const float ik = 1.f / fmaxf(sqrtf(nk), kNormEps);
            float pq = 0.f, pk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xq[e] *= iq;   // normalised rows
                xk[e] *= ik;
                pq = fmaf(xq[e], sq[e], pq);
                pk = fmaf(xk[e], sk[e], pk);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                pq += __shfl_xor_sync(0xffffffffu, pq, off);
                pk += __shfl_xor_sync(0xffffffffu, pk, off);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq[e] = (sq[e] - xq[e] * pq) * iq;
                sk[e] = (sk[e] - xk[e] * pk) * ik;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = lane + 32 * e;
            if (c < d.K) {
                dq[row * d.K + c] = from_f<Tin>(sq[e]);
                dk[row * d.K + c] = from_f<Tin>(sk[e]);
            }
        }
    }
}

// Chunk table of packed variable-length sequences.  Sequence s spans tokens
// [cu[s], cu[s+1]) and is cut into ceil(len / C) chunks, the last one
// partial.  cu must start at 0, end at T and not decrease; then the chunks
// number at most ceil(T / C) + nseq = NT.  Otherwise the error is recorded in
// g_simt_error (reported by kda_check) and no sequence gets a chunk, so no
// kernel reads or writes out of bounds.  One block: thread 0 checks cu and
// forms the prefix of the chunk counts, all threads fill the table.
__device__ int g_simt_error = 0;

__global__ void varlen_table_kernel(const int* __restrict__ cu, int nseq, int T, int C, int NT,
                                    int* __restrict__ ctab, int* __restrict__ sfirst) {
    if (threadIdx.x == 0) {
        bool ok = cu[0] == 0 && cu[nseq] == T;
        for (int s = 0; s < nseq; ++s) ok = ok && cu[s + 1] >= cu[s];
        int total = 0;
        for (int s = 0; s < nseq; ++s) {
            sfirst[s] = total;
            if (ok) total += (cu[s + 1] - cu[s] + C - 1) / C;
        }
        sfirst[nseq] = total;
        if (!ok) atomicCAS(&g_simt_error, 0, 1);
    }
    __syncthreads();
    for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
        const int first = sfirst[s], end = sfirst[s + 1];   // empty unless cu is valid
        for (int j = first; j < end; ++j) {
            const int t0 = cu[s] + (j - first) * C;
            ctab[2 * j] = t0;
            ctab[2 * j + 1] = min(C, cu[s + 1] - t0);
        }
    }
    for (int j = sfirst[nseq] + threadIdx.x; j < NT; j += blockDim.x) {
        ctab[2 * j] = 0;
        ctab[2 * j + 1] = 0;
    }
}

template <typename F>
kda_status set_smem(F* kernel, size_t bytes) {
    if (bytes > 227 * 1024) return KDA_ERR_UNSUPPORTED;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

template <typename Tin>
kda_status run_intra(const Dims& d, const Ws& w, const void* q, const void* k, const void* v,
                     const void* g, const void* beta, cudaStream_t s) {
    kda_status st;
    const size_t si = intra_smem(d);
    auto intra = d.C > 64 ? intra_kernel<Tin, true> : intra_kernel<Tin, false>;
    if ((st = set_smem(intra, si)) != KDA_OK) return st;
    {
        TimedLaunch tl("simt_intra", s);
        intra<<<dim3(d.NT, d.B * d.HV), kThreads, si, s>>>(
            d, w, static_cast<const Tin*>(q), static_cast<const Tin*>(k),
            static_cast<const Tin*>(v), static_cast<const Tin*>(g), static_cast<const Tin*>(beta));
    }
    return launch_status();
}

template <typename Tin>
kda_status run_forward_parts(const Dims& d, const Ws& w, const void* q, const void* k,
                             const void* v, const void* g, const void* beta, const float* h0,
                             void* o, float* ht, int mode, cudaStream_t s) {
    kda_status st = run_intra<Tin>(d, w, q, k, v, g, beta, s);
    if (st != KDA_OK) return st;
    const size_t sf = statef_smem(d);
    auto statef = d.C > 64 ? state_fwd_kernel<Tin, true> : state_fwd_kernel<Tin, false>;
    if ((st = set_smem(statef, sf)) != KDA_OK) return st;
    {
        TimedLaunch tl("simt_state_fwd", s);
        statef<<<dim3((d.V + kVT - 1) / kVT, d.NS), kThreads, sf, s>>>(
            d, w, h0, static_cast<Tin*>(o), ht, mode);
    }
    return launch_status();
}

}  // namespace

size_t simt_workspace_bytes(const kda_dims& kd, int for_bwd) {
    return carve(make_dims(kd), for_bwd, nullptr, nullptr);
}

kda_status simt_fwd(const kda_dims& kd, const void* q, const void* k, const void* v,
                    const void* g, const void* beta, const float* h0, void* o, float* ht,
                    void* ws, cudaStream_t s) {
    const Dims d = make_dims(kd);
    Ws w;
    carve(d, 0, static_cast<char*>(ws), &w);
    if (kd.dtype == KDA_BF16)
        return run_forward_parts<__nv_bfloat16>(d, w, q, k, v, g, beta, h0, o, ht, 1, s);
    return run_forward_parts<float>(d, w, q, k, v, g, beta, h0, o, ht, 1, s);
}

namespace {
template <typename Tin>
kda_status simt_tail_t(const Dims& d, const Ws& w, const void* q, const void* k, const void* g,
                       const void* beta, void* dq, void* dk, void* dg, void* dbeta,
                       cudaStream_t s) {
    kda_status st;
    const size_t sk = kgrad_smem(d);
    auto kgrad = d.C > 64 ? kgrad_kernel<Tin, true> : kgrad_kernel<Tin, false>;
    if ((st = set_smem(kgrad, sk)) != KDA_OK) return st;
    const int BH = d.B * d.HV;
    {
        TimedLaunch tl("simt_kgrad", s);
        kgrad<<<dim3(d.NT, BH), kThreads, sk, s>>>(
            d, w, static_cast<const Tin*>(q), static_cast<const Tin*>(k),
            static_cast<const Tin*>(g), static_cast<const Tin*>(beta), static_cast<Tin*>(dg),
            static_cast<Tin*>(dbeta));
    }
    if ((st = launch_status()) != KDA_OK) return st;
    const size_t rows = (size_t)d.B * d.Tr * d.H;
    const int nblk = (int)std::min<size_t>((rows + 7) / 8, 152 * 16);
    if (nblk == 0) return KDA_OK;
    {
        TimedLaunch tl("simt_group_sum", s);
        group_sum_kernel<Tin><<<nblk, 256, 0, s>>>(d, w.dqh, w.dkh, static_cast<const Tin*>(q),
                                                   static_cast<const Tin*>(k),
                                                   static_cast<Tin*>(dq), static_cast<Tin*>(dk));
    }
    return launch_status();
}

template <typename Tin>
kda_status simt_bwd_t(const Dims& d, const Ws& w, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, const float* h0, const void* dout,
                      const float* dht, void* dq, void* dk, void* dv, void* dg, void* dbeta,
                      float* dh0, cudaStream_t s) {
    kda_status st = run_forward_parts<Tin>(d, w, q, k, v, g, beta, h0, nullptr, nullptr, 2, s);
    if (st != KDA_OK) return st;
    const size_t sb = statef_smem(d), sv = vgrad_smem(d);
    auto stateb = d.C > 64 ? state_bwd_kernel<Tin, true> : state_bwd_kernel<Tin, false>;
    auto vgrad = d.C > 64 ? vgrad_kernel<Tin, true> : vgrad_kernel<Tin, false>;
    if ((st = set_smem(stateb, sb)) != KDA_OK) return st;
    if ((st = set_smem(vgrad, sv)) != KDA_OK) return st;
    const int BH = d.B * d.HV;
    {
        TimedLaunch tl("simt_state_bwd", s);
        stateb<<<dim3((d.V + kVT - 1) / kVT, d.NS), kThreads, sb, s>>>(
            d, w, static_cast<const Tin*>(dout), dht, dh0);
    }
    if ((st = launch_status()) != KDA_OK) return st;
    {
        TimedLaunch tl("simt_vgrad", s);
        vgrad<<<dim3(d.NT, BH), kThreads, sv, s>>>(
            d, w, static_cast<const Tin*>(v), static_cast<const Tin*>(beta),
            static_cast<const Tin*>(dout), static_cast<Tin*>(dv));
    }
    if ((st = launch_status()) != KDA_OK) return st;
    return simt_tail_t<Tin>(d, w, q, k, g, beta, dq, dk, dg, dbeta, s);
}
}  // namespace

namespace {
// Kernel dims of a packed variable-length batch: B = 1, T padded to the
// chunk-table bound ceil(T / C) + nseq chunks, Tr the real token count.
Dims varlen_dims(const kda_dims& kd, int nseq) {
    Dims d = make_dims(kd);
    d.NT = (kd.T + d.C - 1) / d.C + nseq;
    d.T = d.NT * d.C;
    d.Tr = kd.T;
    d.NS = nseq * d.HV;
    return d;
}

// The SIMT workspace of the padded batch, then the chunk table [NT][2] and
// the sequences' first chunks [nseq + 1].
size_t varlen_carve(const kda_dims& kd, int nseq, int for_bwd, char* base, Ws* w, Dims* out) {
    Dims d = varlen_dims(kd, nseq);
    size_t off = carve(d, for_bwd, base, w);
    int* ctab = base ? reinterpret_cast<int*>(base + off) : nullptr;
    off += align256((size_t)d.NT * 2 * sizeof(int));
    int* sfirst = base ? reinterpret_cast<int*>(base + off) : nullptr;
    off += align256((size_t)(nseq + 1) * sizeof(int));
    d.ctab = ctab;
    d.sfirst = sfirst;
    if (out) *out = d;
    return off;
}

kda_status varlen_table(const Dims& d, const int* cu, int nseq, cudaStream_t s) {
    varlen_table_kernel<<<1, 256, 0, s>>>(cu, nseq, d.Tr, d.C, d.NT, const_cast<int*>(d.ctab),
                                          const_cast<int*>(d.sfirst));
    return launch_status();
}
}  // namespace

kda_status varlen_table_launch(const int* cu, int nseq, int T, int C, int NT, int* ctab,
                               int* sfirst, cudaStream_t s) {
    varlen_table_kernel<<<1, 256, 0, s>>>(cu, nseq, T, C, NT, ctab, sfirst);
    return launch_status();
}

size_t simt_varlen_workspace_bytes(const kda_dims& kd, int nseq, int for_bwd) {
    return varlen_carve(kd, nseq, for_bwd, nullptr, nullptr, nullptr);
}

kda_status simt_fwd_varlen(const kda_dims& kd, const int* cu, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const float* h0, void* o, float* ht, void* ws, cudaStream_t s) {
    Ws w;
    Dims d;
    varlen_carve(kd, nseq, 0, static_cast<char*>(ws), &w, &d);
    kda_status st = varlen_table(d, cu, nseq, s);
    if (st != KDA_OK) return st;
    if (kd.dtype == KDA_BF16)
        return run_forward_parts<__nv_bfloat16>(d, w, q, k, v, g, beta, h0, o, ht, 1, s);
    return run_forward_parts<float>(d, w, q, k, v, g, beta, h0, o, ht, 1, s);
}

kda_status simt_bwd_varlen(const kda_dims& kd, const int* cu, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const void* beta,
                           const float* h0, const void* dout, const float* dht, void* dq,
                           void* dk, void* dv, void* dg, void* dbeta, float* dh0, void* ws,
                           cudaStream_t s) {
    Ws w;
    Dims d;
    varlen_carve(kd, nseq, 1, static_cast<char*>(ws), &w, &d);
    kda_status st = varlen_table(d, cu, nseq, s);
    if (st != KDA_OK) return st;
    if (kd.dtype == KDA_BF16)
        return simt_bwd_t<__nv_bfloat16>(d, w, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg,
                                         dbeta, dh0, s);
    return simt_bwd_t<float>(d, w, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0,
                             s);
}

kda_status simt_take_error(cudaStream_t s) {
    int err = 0;
    if (cudaMemcpyFromSymbolAsync(&err, g_simt_error, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                  s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (err == 0) return KDA_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_simt_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    cudaStreamSynchronize(s);
    return KDA_ERR_SHAPE;
}

kda_status group_sum_launch(const kda_dims& kd, const float* dqh, const float* dkh,
                            const void* q, const void* k, void* dq, void* dk, cudaStream_t s) {
    const Dims d = make_dims(kd);
    const size_t rows = (size_t)d.B * d.T * d.H;
    const int nblk = (int)std::min<size_t>((rows + 7) / 8, 152 * 16);
    TimedLaunch tl("group_sum", s);
    if (kd.dtype == KDA_BF16)
        group_sum_kernel<__nv_bfloat16><<<nblk, 256, 0, s>>>(
            d, dqh, dkh, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk));
    else
        group_sum_kernel<float><<<nblk, 256, 0, s>>>(d, dqh, dkh, static_cast<const float*>(q),
                                                     static_cast<const float*>(k),
                                                     static_cast<float*>(dq),
                                                     static_cast<float*>(dk));
    return launch_status();
}

void simt_ws_ptrs(const kda_dims& kd, int for_bwd, void* ws, SimtWsPtrs* o) {
    const Dims d = make_dims(kd);
    Ws w;
    carve(d, for_bwd, static_cast<char*>(ws), &w);
    o->W = w.W; o->U = w.U; o->Qh = w.Qh; o->Kb = w.Kb; o->Aqk = w.Aqk; o->Tm = w.Tm;
    o->gam = w.gam; o->dlt = w.dlt; o->hs = w.hs; o->dhs = w.dhs; o->ddl = w.ddl;
    o->dQh = w.dQh; o->dWm = w.dWm; o->dKb = w.dKb; o->dgam = w.dgam; o->dAqk = w.dAqk;
    o->dTv = w.dTv; o->dbv = w.dbv; o->dqh = w.dqh; o->dkh = w.dkh;
}

kda_status simt_bwd(const kda_dims& kd, const void* q, const void* k, const void* v,
                    const void* g, const void* beta, const float* h0, const void* dout,
                    const float* dht, void* dq, void* dk, void* dv, void* dg, void* dbeta,
                    float* dh0, void* ws, cudaStream_t s) {
    const Dims d = make_dims(kd);
    Ws w;
    carve(d, 1, static_cast<char*>(ws), &w);
    if (kd.dtype == KDA_BF16)
        return simt_bwd_t<__nv_bfloat16>(d, w, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg,
                                         dbeta, dh0, s);
    return simt_bwd_t<float>(d, w, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0,
                             s);
}

}  // namespace kda
