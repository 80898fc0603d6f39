// Chunk-local part of the backward for K = V = 128, chunk 64: register-tiled
// fp32 CUDA-core kernel, one CTA (512 threads) per (chunk, head).
//
// Inputs per chunk (fp32 workspace, written by the V-contraction kernel and
// the intra-chunk kernel): T, dW, dQh, dKb, dAqk, dTv, dgam, dbv; and q, k,
// g, beta.  With G_r the in-chunk cumsum of max(g,-5), khat = k o exp(G),
// Y = diag(beta) khat:
//     dT   = mask_strict(diag(beta) dTv + dW Y^T)            (dT_im uses beta_m)
//     dKb' = T^T dW              (gradient of beta khat)
//     dA   = -mask_strict(T^T (dT T^T))
//     sA   = sum_{j<r} dA[r][j] k_j e(r,j),    sQ = sum_{j<=r} dAqk[r][j] k_j e(r,j)
//     cA   = sum_{t>r} dA[t][r] beta_t k_t e(t,r),  cQ = sum_{t>=r} dAqk[t][r] qs_t e(t,r)
//   with e(t,j) = exp(G_t - G_j) factored per 16-row block (reference row b):
//   e(t,j) = E_t F[R(t)][R(j)] / E_j, E_r = exp(G_r - G_b(r)) in [e^-75, 1].
//     dk  = beta dKb' e^G + dKb e^{G_last-G} + beta sA + cA + cQ
//     dqs = dQh e^G + sQ
//     dG  = beta k dKb' e^G + qs dQh e^G - k dKb e^{G_last-G} + beta k sA + qs sQ - k (cA+cQ)
//           (+ sum_r dKb_r Kb_r + dgam gam on the last row)
//     dbeta = dbv + sum_c (dKb' k e^G + k sA)
//     dg_s  = [g_s >= -5] sum_{r>=s} dG_r,   dq = scale dqs
// Thread (tr, tc) = (tid / 32, tid % 32) owns rows 4tr..4tr+3 and columns
// tc + 32j of every 64 x 128 result (and columns tc, tc+32 of 64 x 64 ones),
// so each reduction step loads 4 broadcast row values and a few
// conflict-free column values for 8-16 independent FMAs.  The fp32 inputs
// arrive with asynchronous 4-byte copies (many in flight per thread).
#include "kda_common.cuh"
#include "kda_timing.cuh"

namespace kda {
namespace {

constexpr int C = 64, K = 128, KP = K + 1, CP = C + 1, NTH = 512, RPT = 4;

struct LocalArgs {
    int T, H, HV, NT, G;
    float scale;
    const float *Tm, *dW, *dQh, *dKb, *dAqk, *dTv, *dgam, *dbv;
    float *dqh, *dkh;  // fp32 per-value-head outputs (used when G > 1)
};

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename Tin>
__global__ void __launch_bounds__(NTH, 1)
local_bwd_kernel(LocalArgs a, const Tin* __restrict__ q, const Tin* __restrict__ k,
                 const Tin* __restrict__ g, const Tin* __restrict__ beta, Tin* __restrict__ dq,
                 Tin* __restrict__ dk, Tin* __restrict__ dg, Tin* __restrict__ dbeta) {
    extern __shared__ float sm[];
    float* kS = sm;              // k
    float* qS = kS + C * KP;     // scale * q
    float* GS = qS + C * KP;     // cumsum of clamped g
    float* X = GS + C * KP;      // dW, then KE = k / E, then KLb = beta k E
    float* Y = X + C * KP;       // beta khat, then dKb', then QL = qs E
    float* Ts = Y + C * KP;      // T
    float* D = Ts + C * CP;      // dT, then dT T^T, then dA
    float* Aq = D + C * CP;      // dAqk
    float* bS = Aq + C * CP;     // beta
    float* Fb = bS + C;          // F[fidx(R,J)][c]
    float* eGb = Fb + 10 * K;    // exp(G_bR)
    float* eLb = eGb + 4 * K;    // exp(G_last - G_bR)

    const int tid = threadIdx.x, tr = tid >> 5, tc = tid & 31;
    const int n = blockIdx.x, bh = blockIdx.y;
    const int b = bh / a.HV, hv = bh % a.HV, h = hv / a.G;
    const int t0 = n * C;
    const size_t row0 = (size_t)bh * a.T + t0;
    const size_t cc0 = ((size_t)bh * a.NT + n) * C * C;
    auto tok = [&](int r, int head, int nheads) {
        return (((size_t)b * a.T + t0 + r) * nheads + head) * K;
    };
    auto fidx = [](int R, int J) { return R * (R + 1) / 2 + J; };

    // ---- load: fp32 arrays asynchronously, bf16 inputs converted ----
    for (int i = tid; i < C * K; i += NTH) {
        const int r = i / K, c = i % K;
        cp_async4(&X[r * KP + c], &a.dW[(row0 + r) * K + c]);
    }
    for (int i = tid; i < C * C; i += NTH) {
        const int r = i / C, c = i % C;
        cp_async4(&Ts[r * CP + c], &a.Tm[cc0 + i]);
        cp_async4(&Aq[r * CP + c], &a.dAqk[cc0 + i]);
    }
#pragma unroll 4
    for (int i = tid; i < C * K; i += NTH) {
        const int r = i / K, c = i % K;
        kS[r * KP + c] = to_f(k[tok(r, h, a.H) + c]);
        qS[r * KP + c] = a.scale * to_f(q[tok(r, h, a.H) + c]);
        GS[r * KP + c] = fmaxf(to_f(g[tok(r, hv, a.HV) + c]), kGateFloor);
    }
    cp_async_wait_all();
    if (tid < C) bS[tid] = to_f(beta[((size_t)b * a.T + t0 + tid) * a.HV + hv]);
    __syncthreads();
    if (tid < K) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += GS[r * KP + tid];
            GS[r * KP + tid] = acc;
        }
    }
    __syncthreads();
    for (int i = tid; i < C * K; i += NTH) {
        const int r = i / K, c = i % K;
        Y[r * KP + c] = bS[r] * kS[r * KP + c] * __expf(GS[r * KP + c]);
    }
    for (int i = tid; i < 16 * K; i += NTH) {
        const int R = i / (4 * K), J = (i / K) % 4, c = i % K;
        if (J <= R) Fb[fidx(R, J) * K + c] = __expf(GS[16 * R * KP + c] - GS[16 * J * KP + c]);
    }
    for (int i = tid; i < 4 * K; i += NTH) {
        const int R = i / K, c = i % K;
        eGb[i] = __expf(GS[16 * R * KP + c]);
        eLb[i] = __expf(GS[(C - 1) * KP + c] - GS[16 * R * KP + c]);
    }
    __syncthreads();

    const int r0 = RPT * tr;
    // ---- dT = mask_strict(beta_m dTv + dW Y^T)  (64 x 64; cols tc, tc+32) ----
    {
        float acc[RPT][2];
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
        for (int c = 0; c < K; ++c) {
            const float y0 = Y[tc * KP + c], y1 = Y[(tc + 32) * KP + c];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float x = X[(r0 + i) * KP + c];
                acc[i][0] += x * y0;
                acc[i][1] += x * y1;
            }
        }
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int ii = r0 + i, m = tc + 32 * u;
                D[ii * CP + m] = m < ii ? bS[m] * a.dTv[cc0 + ii * C + m] + acc[i][u] : 0.f;
            }
    }
    __syncthreads();
    // ---- dKb' = T^T dW  (64 x 128) -> Y ----
    {
        float acc[RPT][4];
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[i][u] = 0.f;
#pragma unroll 2
        for (int rr = 0; rr < C; ++rr) {
            float xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) xv[u] = X[rr * KP + tc + 32 * u];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float tv = Ts[rr * CP + r0 + i];  // T[rr][m], zero for rr < m
#pragma unroll
                for (int u = 0; u < 4; ++u) acc[i][u] += tv * xv[u];
            }
        }
        __syncthreads();  // Y (beta khat) fully consumed by dT above
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) Y[(r0 + i) * KP + tc + 32 * u] = acc[i][u];
    }
    // ---- Y2 = dT T^T, then dA = -mask_strict(T^T Y2)  (in D) ----
    {
        float acc[RPT][2];
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
        for (int m = 0; m < C; ++m) {
            const float t0v = Ts[tc * CP + m], t1v = Ts[(tc + 32) * CP + m];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float dv = D[(r0 + i) * CP + m];
                acc[i][0] += dv * t0v;
                acc[i][1] += dv * t1v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            D[(r0 + i) * CP + tc] = acc[i][0];
            D[(r0 + i) * CP + tc + 32] = acc[i][1];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
        for (int m = 0; m < C; ++m) {
            const float y0 = D[m * CP + tc], y1 = D[m * CP + tc + 32];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float tv = Ts[m * CP + r0 + i];  // T[m][i]
                acc[i][0] += tv * y0;
                acc[i][1] += tv * y1;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int ii = r0 + i, j = tc + 32 * u;
                D[ii * CP + j] = j < ii ? -acc[i][u] : 0.f;
            }
    }
    // ---- row-side table X <- KE = k / E ----
    for (int i = tid; i < C * K; i += NTH) {
        const int r = i / K, c = i % K;
        X[r * KP + c] = kS[r * KP + c] * __expf(GS[(r & ~15) * KP + c] - GS[r * KP + c]);
    }
    __syncthreads();

    // ---- row side: sA, sQ for rows r0..r0+RPT-1 (one 16-row block R) ----
    const int R = r0 >> 4;
    float sA[RPT][4], sQ[RPT][4];
    {
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) sA[i][u] = sQ[i][u] = 0.f;
        for (int J = 0; J <= R; ++J) {
            float pa[RPT][4], pq[RPT][4];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int u = 0; u < 4; ++u) pa[i][u] = pq[i][u] = 0.f;
#pragma unroll 2
            for (int j = 16 * J; j < 16 * J + 16; ++j) {
                float ke[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) ke[u] = X[j * KP + tc + 32 * u];
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float da = D[(r0 + i) * CP + j], dq_ = Aq[(r0 + i) * CP + j];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        pa[i][u] += da * ke[u];
                        pq[i][u] += dq_ * ke[u];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float f = Fb[fidx(R, J) * K + tc + 32 * u];
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    sA[i][u] += f * pa[i][u];
                    sQ[i][u] += f * pq[i][u];
                }
            }
        }
    }
    __syncthreads();
    // ---- column-side tables: X <- KLb = beta k E, qS <- QL = qs E ----
    // (the assembly below recovers qs = QL / E)
    for (int i = tid; i < C * K; i += NTH) {
        const int r = i / K, c = i % K;
        const float E = __expf(GS[r * KP + c] - GS[(r & ~15) * KP + c]);
        X[r * KP + c] = bS[r] * kS[r * KP + c] * E;
        qS[r * KP + c] *= E;
    }
    __syncthreads();
    float cAQ[RPT][4];
    {
        const int J = R;
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) cAQ[i][u] = 0.f;
        for (int RR = J; RR < 4; ++RR) {
            float pa[RPT][4];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int u = 0; u < 4; ++u) pa[i][u] = 0.f;
#pragma unroll 2
            for (int t = 16 * RR; t < 16 * RR + 16; ++t) {
                float kl[4], ql[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = tc + 32 * u;
                    kl[u] = X[t * KP + c];
                    ql[u] = qS[t * KP + c];
                }
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float da = D[t * CP + r0 + i], dq_ = Aq[t * CP + r0 + i];
#pragma unroll
                    for (int u = 0; u < 4; ++u) pa[i][u] += da * kl[u] + dq_ * ql[u];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float f = Fb[fidx(RR, J) * K + tc + 32 * u];
#pragma unroll
                for (int i = 0; i < RPT; ++i) cAQ[i][u] += f * pa[i][u];
            }
        }
    }
    __syncthreads();

    // ---- assemble per element; dG into X, dbeta partials into GS? (GS still needed) ----
    // dG -> X (KLb no longer needed), dbeta partial -> D rows? use Aq-free space: reuse Ts.
    float dGv[RPT][4], dbp[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) dbp[i] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = r0 + i;
        const float br = bS[r];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = tc + 32 * u;
            const float G = GS[r * KP + c];
            const float E = __expf(G - GS[(r & ~15) * KP + c]);
            const float Einv = 1.f / E;
            const float eG = eGb[R * K + c] * E;
            const float eL = eLb[R * K + c] * Einv;
            const float kr = kS[r * KP + c], qr = qS[r * KP + c] * Einv;  // QL / E
            const float dKbeta = Y[r * KP + c];
            const float dQh = a.dQh[(row0 + r) * K + c];
            const float dKb = a.dKb[(row0 + r) * K + c];
            const float sa = sA[i][u] * E, sq = sQ[i][u] * E;
            const float caq = cAQ[i][u] * Einv;
            const float dkv = br * dKbeta * eG + dKb * eL + br * sa + caq;
            const float dqs = dQh * eG + sq;
            dGv[i][u] = dKbeta * br * kr * eG + dQh * qr * eG - dKb * kr * eL + br * kr * sa +
                        qr * sq - kr * caq;
            dbp[i] += dKbeta * kr * eG + kr * sa;
            if (a.G == 1) {
                dq[tok(r, hv, a.HV) + c] = from_f<Tin>(a.scale * dqs);
                dk[tok(r, hv, a.HV) + c] = from_f<Tin>(dkv);
            } else {
                a.dqh[tok(r, hv, a.HV) + c] = a.scale * dqs;
                a.dkh[tok(r, hv, a.HV) + c] = dkv;
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) X[(r0 + i) * KP + tc + 32 * u] = dGv[i][u];
    // dbeta: reduce the 32 column groups of each row with warp shuffles
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        float v = dbp[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (tc == 0) {
            const int r = r0 + i;
            dbeta[((size_t)b * a.T + t0 + r) * a.HV + hv] = from_f<Tin>(v + a.dbv[row0 + r]);
        }
    }
    __syncthreads();
    // last-row terms and dg = [g >= -5] reverse cumsum of dG
    if (tid < K) {
        const int c = tid;
        const float gl = GS[(C - 1) * KP + c];
        float acc = a.dgam[((size_t)bh * a.NT + n) * K + c] * __expf(gl);
        for (int r = 0; r < C; ++r)
            acc += a.dKb[(row0 + r) * K + c] * kS[r * KP + c] * __expf(gl - GS[r * KP + c]);
        X[(C - 1) * KP + c] += acc;
        float run = 0.f;
        for (int r = C - 1; r >= 0; --r) {
            run += X[r * KP + c];
            const size_t ig = tok(r, hv, a.HV) + c;
            dg[ig] = from_f<Tin>(to_f(g[ig]) >= kGateFloor ? run : 0.f);
        }
    }
}

size_t local_smem() {
    return sizeof(float) * (5 * (size_t)C * KP + 3 * (size_t)C * CP + C + 18 * K);
}

}  // namespace

kda_status local_bwd_launch(const kda_dims& d, const SimtWsPtrs& p, const void* q,
                            const void* k, const void* g, const void* beta, void* dq, void* dk,
                            void* dg, void* dbeta, cudaStream_t s) {
    if (d.dtype != KDA_BF16 || d.K != K || d.V != K || d.chunk_size != C)
        return KDA_ERR_UNSUPPORTED;
    LocalArgs a;
    a.T = d.T;
    a.H = d.H;
    a.HV = d.HV;
    a.NT = d.T / C;
    a.G = d.HV / d.H;
    a.scale = d.scale;
    a.Tm = p.Tm;
    a.dW = p.dWm;
    a.dQh = p.dQh;
    a.dKb = p.dKb;
    a.dAqk = p.dAqk;
    a.dTv = p.dTv;
    a.dgam = p.dgam;
    a.dbv = p.dbv;
    a.dqh = p.dqh;
    a.dkh = p.dkh;
    const size_t smem = local_smem();
    if (cudaFuncSetAttribute(local_bwd_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return KDA_ERR_CUDA;
    {
        TimedLaunch tl("local_bwd", s);
        local_bwd_kernel<__nv_bfloat16><<<dim3(a.NT, d.B * d.HV), NTH, smem, s>>>(
            a, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(beta),
            static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
            static_cast<__nv_bfloat16*>(dg), static_cast<__nv_bfloat16*>(dbeta));
    }
    return launch_status();
}

}  // namespace kda
