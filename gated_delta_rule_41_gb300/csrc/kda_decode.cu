// Single-token KDA decode step (K3 README, table 实现路线表, row L6: recurrent
// decode on a KDAState [B,HV,K,V]; row L1 gives the per-token formula).
//
// Per head, with a = exp(max(g,-5)) and qs = scale*q, the update needs two
// reductions over K of the OLD state only:
//     sk = (a o k)^T S,   sq = (a o qs)^T S          (V-vectors)
//     e  = v - sk
//     o  = sq + beta (k . qs) e                       (= S_new^T qs)
//     S_new = diag(a) S + beta k e^T
// so the state is read once and written once.  The kernel holds its slice of
// S in registers between the read and the write, streams it with 128-bit
// evict-first loads/stores, and reduces the column sums through shared
// memory.  HBM traffic per head: 2*K*V*4 bytes of state plus the token vectors.
#include "kda_common.cuh"
#include "kda_timing.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

constexpr float kNormEps = 1e-12f;

// Fast path: K, V multiples of 4.  A CTA takes VT of a head's V value
// columns (the columns are independent: each one's reductions over K and
// its update touch only that column), with (VT/4) threads per state row;
// each thread owns 4 consecutive columns of ROWS rows.  QKN: q and k are
// L2-normalised over K first (x / max(|x|, 1e-12)).  Each CTA alternates a
// load, a reduction and a store phase; with VT = 32 a thread holds 16 (K =
// 128) or 8 (K = 64) floats of state and six CTAs share an SM, so more of
// the state stays in flight than with a whole head per CTA.
template <typename Tin, int K, int V, bool QKN, int VT = V>
__global__ void __launch_bounds__(kDecodeThreads, VT == V ? 3 : (VT >= 64 ? 5 : 6))
decode_kernel(int H, int HV, float scale, const Tin* __restrict__ q, const Tin* __restrict__ k,
              const Tin* __restrict__ v, const Tin* __restrict__ g,
              const Tin* __restrict__ beta, float* __restrict__ state, Tin* __restrict__ o) {
    constexpr int NVT = V / VT;                 // CTAs per head
    constexpr int TPR = VT / 4;                 // threads per state row
    constexpr int RS = V / 4;                   // float4 per state row
    constexpr int RP = kDecodeThreads / TPR;    // rows per pass
    constexpr int ROWS = K / RP;                // rows per thread
    static_assert(V % VT == 0 && VT % 4 == 0, "bad value tile");
    static_assert(kDecodeThreads % TPR == 0 && K % RP == 0, "bad decode tiling");

    __shared__ float s_qa[K], s_ka[K], s_a[K], s_k[K];
    __shared__ float s_red[2][RP][VT];
    __shared__ float s_e[VT];
    __shared__ float s_kq[K / 32];
    __shared__ float s_nk[K / 32], s_nq[K / 32];

    const int bh = blockIdx.x / NVT, v0 = (blockIdx.x % NVT) * VT;
    const int b = bh / HV, hv = bh % HV, h = hv / (HV / H);
    const int tid = threadIdx.x;
    const int col4 = tid % TPR;
    const int row0 = tid / TPR;

    float4* S4 = reinterpret_cast<float4*>(state + (size_t)bh * K * V + v0);
    float4 s[ROWS];
#pragma unroll
    for (int i = 0; i < ROWS; ++i) s[i] = __ldcs(S4 + (size_t)(row0 + i * RP) * RS + col4);

    const size_t qk_off = ((size_t)b * H + h) * K;
    float kk = 0.f, qq = 0.f;
    if (QKN) {
        if (tid < K) {
            kk = to_f(k[qk_off + tid]);
            qq = to_f(q[qk_off + tid]);
            float nk = kk * kk, nq = qq * qq;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                nk += __shfl_xor_sync(0xffffffffu, nk, off);
                nq += __shfl_xor_sync(0xffffffffu, nq, off);
            }
            if ((tid & 31) == 0) {
                s_nk[tid >> 5] = nk;
                s_nq[tid >> 5] = nq;
            }
        }
        __syncthreads();
        if (tid < K) {
            float nk = 0.f, nq = 0.f;
#pragma unroll
            for (int w = 0; w < K / 32; ++w) {
                nk += s_nk[w];
                nq += s_nq[w];
            }
            kk *= 1.f / fmaxf(sqrtf(nk), kNormEps);
            qq *= scale / fmaxf(sqrtf(nq), kNormEps);
        }
    }
    if (tid < K) {  // K is a multiple of 32: these warps are fully active
        const float a = __expf(fmaxf(to_f(g[(size_t)bh * K + tid]), kGateFloor));
        if (!QKN) {
            kk = to_f(k[qk_off + tid]);
            qq = scale * to_f(q[qk_off + tid]);
        }
        s_a[tid] = a;
        s_k[tid] = kk;
        s_ka[tid] = a * kk;
        s_qa[tid] = a * qq;
        float kq = kk * qq;  // k . qs, per warp
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if ((tid & 31) == 0) s_kq[tid >> 5] = kq;
    }
    __syncthreads();

    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        const int c = row0 + i * RP;
        const float ka = s_ka[c], qa = s_qa[c];
        pk.x += ka * s[i].x; pk.y += ka * s[i].y; pk.z += ka * s[i].z; pk.w += ka * s[i].w;
        pq.x += qa * s[i].x; pq.y += qa * s[i].y; pq.z += qa * s[i].z; pq.w += qa * s[i].w;
    }
    *reinterpret_cast<float4*>(&s_red[0][row0][col4 * 4]) = pk;
    *reinterpret_cast<float4*>(&s_red[1][row0][col4 * 4]) = pq;
    __syncthreads();

    const float bt = to_f(beta[bh]);
    if (tid < VT) {
        float sk = 0.f, sq = 0.f;
#pragma unroll 8
        for (int p = 0; p < RP; ++p) {
            sk += s_red[0][p][tid];
            sq += s_red[1][p][tid];
        }
        float kq = 0.f;
#pragma unroll
        for (int w = 0; w < K / 32; ++w) kq += s_kq[w];
        const float e = to_f(v[(size_t)bh * V + v0 + tid]) - sk;
        s_e[tid] = e;
        o[(size_t)bh * V + v0 + tid] = from_f<Tin>(sq + bt * kq * e);
    }
    __syncthreads();

    const float4 e4 = *reinterpret_cast<const float4*>(&s_e[col4 * 4]);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        const int c = row0 + i * RP;
        const float a = s_a[c], bk = bt * s_k[c];
        float4 r;
        r.x = a * s[i].x + bk * e4.x;
        r.y = a * s[i].y + bk * e4.y;
        r.z = a * s[i].z + bk * e4.z;
        r.w = a * s[i].w + bk * e4.w;
        __stcs(S4 + (size_t)c * RS + col4, r);
    }
}

// Any K, V <= 128: one thread per value column, two passes over the state.
template <typename Tin>
__global__ void __launch_bounds__(128)
decode_kernel_generic(int H, int HV, int K, int V, float scale, int qkn, const Tin* __restrict__ q,
                      const Tin* __restrict__ k, const Tin* __restrict__ v,
                      const Tin* __restrict__ g, const Tin* __restrict__ beta,
                      float* __restrict__ state, Tin* __restrict__ o) {
    __shared__ float s_a[128], s_k[128], s_q[128];
    const int bh = blockIdx.x;
    const int b = bh / HV, hv = bh % HV, h = hv / (HV / H);
    const int j = threadIdx.x;
    const size_t qk_off = ((size_t)b * H + h) * K;
    for (int c = j; c < K; c += blockDim.x) {
        s_a[c] = expf(fmaxf(to_f(g[(size_t)bh * K + c]), kGateFloor));
        s_k[c] = to_f(k[qk_off + c]);
        s_q[c] = scale * to_f(q[qk_off + c]);
    }
    __syncthreads();
    float ik = 1.f, iq = 1.f;   // with qkn: the inverse norms of k and q
    if (qkn) {
        float nk = 0.f, nq = 0.f;
        for (int c = 0; c < K; ++c) {
            nk = fmaf(s_k[c], s_k[c], nk);
            nq = fmaf(s_q[c], s_q[c], nq);
        }
        ik = 1.f / fmaxf(sqrtf(nk), kNormEps);
        iq = 1.f / fmaxf(sqrtf(nq) / scale, kNormEps);
    }
    if (j >= V) return;
    float* S = state + (size_t)bh * K * V;
    float sk = 0.f, sq = 0.f, kq = 0.f;
    for (int c = 0; c < K; ++c) {
        const float sv = s_a[c] * S[(size_t)c * V + j];
        sk += s_k[c] * sv;
        sq += s_q[c] * sv;
        kq += s_k[c] * s_q[c];
    }
    sk *= ik;
    sq *= iq;
    kq *= ik * iq;
    const float bt = to_f(beta[bh]);
    const float e = to_f(v[(size_t)bh * V + j]) - sk;
    o[(size_t)bh * V + j] = from_f<Tin>(sq + bt * kq * e);
    for (int c = 0; c < K; ++c) {
        float* p = S + (size_t)c * V + j;
        *p = s_a[c] * *p + bt * (ik * s_k[c]) * e;
    }
}

template <typename Tin>
kda_status decode_dispatch(const kda_dims& d, const void* q, const void* k, const void* v,
                           const void* g, const void* beta, float* state, void* o,
                           cudaStream_t s) {
    const int nb = d.B * d.HV;
    auto* qq = static_cast<const Tin*>(q);
    auto* kk = static_cast<const Tin*>(k);
    auto* vv = static_cast<const Tin*>(v);
    auto* gg = static_cast<const Tin*>(g);
    auto* bb = static_cast<const Tin*>(beta);
    auto* oo = static_cast<Tin*>(o);
    TimedLaunch tl("decode_step", s);
    const bool qkn = d.qk_l2norm != 0;
    if (d.K == 128 && d.V == 128) {
        // four CTAs per head, 32 value columns each
        if (qkn)
            decode_kernel<Tin, 128, 128, true, 32><<<4 * nb, kDecodeThreads, 0, s>>>(
                d.H, d.HV, d.scale, qq, kk, vv, gg, bb, state, oo);
        else
            decode_kernel<Tin, 128, 128, false, 32><<<4 * nb, kDecodeThreads, 0, s>>>(
                d.H, d.HV, d.scale, qq, kk, vv, gg, bb, state, oo);
    } else if (d.K == 64 && d.V == 64) {
        // two CTAs per head, 32 value columns each
        if (qkn)
            decode_kernel<Tin, 64, 64, true, 32><<<2 * nb, kDecodeThreads, 0, s>>>(
                d.H, d.HV, d.scale, qq, kk, vv, gg, bb, state, oo);
        else
            decode_kernel<Tin, 64, 64, false, 32><<<2 * nb, kDecodeThreads, 0, s>>>(
                d.H, d.HV, d.scale, qq, kk, vv, gg, bb, state, oo);
    } else {
        decode_kernel_generic<Tin><<<nb, 128, 0, s>>>(d.H, d.HV, d.K, d.V, d.scale, qkn ? 1 : 0,
                                                      qq, kk, vv, gg, bb, state, oo);
    }
    return launch_status();
}

}  // namespace

kda_status decode_launch(const kda_dims& d, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, float* state, void* o,
                         cudaStream_t s) {
    if (d.dtype == KDA_BF16)
        return decode_dispatch<__nv_bfloat16>(d, q, k, v, g, beta, state, o, s);
    return decode_dispatch<float>(d, q, k, v, g, beta, state, o, s);
}

}  // namespace kda
