// Tensor-core (tcgen05 + TMEM + TMA) chunk scan for bf16, K = V = 128,
// chunk 64.
//
// Forward state pass ("chain") of the chunk form (K3 README, table 实现路线表,
// row L2, step (4): the state passed between chunks).  One CTA per (b, hv)
// walks the chunks in order and keeps the K x V state S on chip, as fp32 in
// tensor memory.  The state products are computed transposed so that the
// MMA M dimension is the value dimension (128 rows = 128 TMEM lanes); the
// output is computed row-major:
//     D12W  = S^T W^T            (M=128 v, N=64 rows, K=128 k)
//     delta^T = U^T - D12W       (epilogue, fp32 -> bf16 operand in smem)
//     O     = Qh S + Aqk delta      (M=128 over the 64 rows of Qh / Aqk and
//                                     64 don't-care rows, N=128 v: row-major)
//     S^T   = diag(gam) S^T + delta^T Kb       (gam applied by the epilogue)
// Per-chunk operands (W, Qh, Kb, Aqk, U as bf16; gam fp32) arrive by TMA
// into a two-stage ring.  Warp roles: warp 0 issues TMA, warp 1 owns TMEM and
// issues MMAs (one thread), warps 2-9 are the epilogue (two threads per TMEM
// lane = value column, each taking half of its columns).  Every mbarrier wait
// is bounded: on expiry the kernel records an error code in g_tc_error and
// unwinds.
#include <algorithm>
#include <mutex>

#include "kda_common.cuh"
#include "kda_ptx.cuh"
#include "kda_timing.cuh"

namespace kda {

__device__ int g_tc_error = 0;

namespace {

using namespace ptx;

constexpr int kC = 64, kD = 128;  // chunk size, K = V
constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz

// ---- error-aware bounded mbarrier wait ----
// Gives up after `limit` cycles (recording `code` in g_tc_error) or as soon
// as another wait has recorded an error.
__device__ __forceinline__ bool wait_bar_limit(uint64_t* bar, uint32_t parity, int code,
                                               long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 255u) == 0) {
            if (*reinterpret_cast<volatile int*>(&g_tc_error) != 0) return false;
            if (clock64() - t0 > limit) {
                atomicCAS(&g_tc_error, 0, code);
                return false;
            }
        }
    }
    return true;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int code) {
    return wait_bar_limit(bar, parity, code, kTimeoutCycles);
}
// Wait for a phase with the time bound only (also after another wait has
// failed), for copies that must land before the CTA exits.
__device__ __forceinline__ void wait_bar_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kTimeoutCycles) return;
}
// Warp-uniform version: every lane waits, the warp proceeds only if all did.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, int code) {
    const bool ok = wait_bar(bar, parity, code);
    return __all_sync(0xffffffffu, ok);
}

// ---- shared-memory plan of the chain kernel (offsets from a 1024-aligned base) ----
constexpr uint32_t OFF_W = 0;          // 64 rows x 128 bf16, 2 k-blocks of 8 KB
constexpr uint32_t OFF_Q = 16384;      // same for Qh
constexpr uint32_t OFF_KBT = 32768;    // Kb: 64 rows (c) x 128 bf16 (k), 2 k-blocks
constexpr uint32_t OFF_AQK = 49152;    // Aqk: 64 rows x 64 bf16
constexpr uint32_t OFF_U = 57344;      // U: 64 x 128 bf16, row-major, unswizzled
constexpr uint32_t STAGE_BYTES = 73728;
constexpr uint32_t STAGE_TX = 16384 * 2 + 16384 + 8192 + 16384 + 512;   // tiles + gam
// S^T operand tiles (128 rows x 128 bf16, 2 k-blocks), one per chunk parity:
// the state store of chunk n may still be reading its tile while the state
// of chunk n + 1 is written to the other
constexpr uint32_t OFF_S = 2 * STAGE_BYTES;
constexpr uint32_t S_TILE = 32768;
constexpr uint32_t OFF_DELTA = OFF_S + 2 * S_TILE;  // delta^T operand: 128 rows x 64 bf16
constexpr uint32_t OFF_GAM = OFF_DELTA + 16384;     // gam (128 fp32) of each stage, 512 B apart
constexpr uint32_t OFF_BAR = OFF_GAM + 1024;
constexpr uint32_t CHAIN_SMEM = OFF_BAR + 256 + 1024;  // + alignment slack
static_assert(CHAIN_SMEM <= 232448, "chain kernels exceed the per-CTA shared memory limit");

// TMA warp, MMA warp, 8 epilogue warps (two per TMEM lane quadrant)
constexpr int kChainThreads = 320, kChainEpi = 256;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_W = 128, TM_O0 = 192, TM_O1 = 320, TM_COLS = 512;

// Sums each of N (16 or 32) per-lane values over the 32 lanes of a warp with
// N - 1 + (32 / N - 1) shuffles (a reduce-scatter butterfly: at offset o a
// lane keeps the half of its remaining values selected by lane bit o and adds
// the partner's copy of that half).  On return lane l holds the warp total of
// value l * N / 32.  v is overwritten.
template <int N>
__device__ __forceinline__ float warp_sum_scatter(float (&v)[N]) {
    static_assert(N == 16 || N == 32, "N must be 16 or 32");
    const int lane = threadIdx.x & 31;
    int o = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return v[0];
}

// eight fp32 <-> eight bf16 (16 bytes)
__device__ __forceinline__ void ld8f(const float* p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}
__device__ __forceinline__ void unpack8(const uint4 v, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
// Low part of a two-term bf16 split, x - bf16(x) rounded to bf16, for 8
// values (the high part is pack8(x), the value the operand tiles hold).
__device__ __forceinline__ uint4 pack8_lo(const float (&x)[8]) {
    float h[8], l[8];
    unpack8(pack8(x), h);
#pragma unroll
    for (int i = 0; i < 8; ++i) l[i] = x[i] - h[i];
    return pack8(l);
}
// Low parts of 32 consecutive values to global memory (16-byte aligned).
__device__ __forceinline__ void store_lo32(__nv_bfloat16* dst, const float (&r)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = r[8 * j + i];
        *reinterpret_cast<uint4*>(dst + 8 * j) = pack8_lo(x);
    }
}

// L2-normalises each of the 64 rows of a [64][128] bf16 token tile (two
// 64-column 128B-swizzled boxes, 8 KB apart) in place: x / max(|x|, 1e-12),
// the squares summed in fp32.  nthreads (256 or 512) threads; sixteen
// consecutive lanes share a row, one 8-channel unit each.
__device__ __forceinline__ void l2norm_tile_rows(uint8_t* tile, int tid, int nthreads) {
    for (int unit = tid; unit < 64 * 16; unit += nthreads) {
        const int row = unit >> 4, o = unit & 15;
        uint4* p = reinterpret_cast<uint4*>(tile + (o >> 3) * 8192 + sw128_offset(row, 8 * (o & 7)));
        float x[8];
        unpack8(*p, x);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= inv;
        *p = pack8(x);
    }
}

// ---- epilogue steps shared by the two chains (thread <-> value column v) ----

__device__ __forceinline__ void store_row_bf16(uint8_t* base, int v, int col0, const float (&r)[32],
                                               float sign) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 pk;
        pk.x = pack_bf16(sign * r[8 * j + 0], sign * r[8 * j + 1]);
        pk.y = pack_bf16(sign * r[8 * j + 2], sign * r[8 * j + 3]);
        pk.z = pack_bf16(sign * r[8 * j + 4], sign * r[8 * j + 5]);
        pk.w = pack_bf16(sign * r[8 * j + 6], sign * r[8 * j + 7]);
        *reinterpret_cast<uint4*>(base + sw128_offset(v, col0 + 8 * j)) = pk;
    }
}

// The chains' epilogue has two threads per value column v (TMEM lane); each
// takes one half of the columns of a step.

// State step, columns k in [64 half, 64 half + 64), in two parts.  First:
// S^T (lane v) from TMEM -- or, for the first chunk, from `init` ([K][V]
// fp32, may be null = zeros) -- into r0, r1 and to k-block `half` of the bf16
// K-major operand tile, then arrive on `bar_tile` (the products that read
// the tile may start).
__device__ __forceinline__ void chain_state_tile(uint32_t tS, uint8_t* tile, bool first,
                                                 const float* init, int D, int v, int half,
                                                 uint64_t* bar_tile, float (&r0)[32],
                                                 float (&r1)[32]) {
    const int k0 = 64 * half;
    if (first) {
        // init is [D][D]: rows and columns at D and beyond are zero
        const bool on = init && v < D && k0 < D;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            r0[i] = on ? init[(size_t)(k0 + i) * D + v] : 0.f;
            r1[i] = on ? init[(size_t)(k0 + 32 + i) * D + v] : 0.f;
        }
    } else {
        tmem_ld32_nw(tS + k0, r0);
        tmem_ld32_nw(tS + k0 + 32, r1);
        tmem_wait_ld_dep(r0);
        tmem_wait_ld_dep(r1);
    }
    uint8_t* kt = tile + 16384 * half;
    store_row_bf16(kt, v, 0, r0, 1.f);
    store_row_bf16(kt, v, 32, r1, 1.f);
    fence_async_smem();
    tc_fence_before();  // earlier TMEM reads of this thread precede the MMAs it releases
    mbar_arrive(bar_tile);
}
// Second part (gam is in the chunk's stage): the TMEM copy is scaled by gam
// (per column k) and stored back, then the thread arrives on `bar_tmem` (the
// products that accumulate into it may start).
__device__ __forceinline__ void chain_state_rescale(uint32_t tS, const float* gam, int half,
                                                    uint64_t* bar_tmem, float (&r0)[32],
                                                    float (&r1)[32]) {
    const int k0 = 64 * half;
    // gam is 16-byte aligned: 16 broadcast float4 loads instead of 64 scalar
    const float4* g4 = reinterpret_cast<const float4*>(gam + k0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 a = g4[i], b = g4[8 + i];
        r0[4 * i] *= a.x;
        r0[4 * i + 1] *= a.y;
        r0[4 * i + 2] *= a.z;
        r0[4 * i + 3] *= a.w;
        r1[4 * i] *= b.x;
        r1[4 * i + 1] *= b.y;
        r1[4 * i + 2] *= b.z;
        r1[4 * i + 3] *= b.w;
    }
    tmem_st32_nw(tS + k0, r0);
    tmem_st32_nw(tS + k0 + 32, r1);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar_tmem);
}

// Delta step, columns c in [32 half, 32 half + 32) of 64: from TMEM (u - D if
// u is given: the 32 values U[c][v], read before the products completed) to
// the bf16 K-major operand tile (negated if `neg_tile`), arrive on bar1 and
// bar2 (if given), then, if `gtile` is given, the true-sign bf16 values into
// it as a 128B-swizzled pair of [64 c][64 v] tiles (for a TMA store).  If
// `glo` is given, the low parts of the true-sign values (x - bf16(x)) go to
// the 32 consecutive bf16 there.
__device__ __forceinline__ void chain_delta_step(uint32_t tD, uint8_t* tile, const float* u,
                                                 bool neg_tile, int v, int half, uint64_t* bar1,
                                                 uint64_t* bar2, uint8_t* gtile,
                                                 __nv_bfloat16* glo = nullptr) {
    const int c0 = 32 * half;
    float d0[32];
    tmem_ld32_nw(tD + c0, d0);
    tmem_wait_ld_dep(d0);
    if (u) {
#pragma unroll
        for (int i = 0; i < 32; ++i) d0[i] = u[i] - d0[i];
    }
    const float sg = neg_tile ? -1.f : 1.f;
    store_row_bf16(tile, v, c0, d0, sg);
    if (glo) store_lo32(glo, d0);
    fence_async_smem();
    tc_fence_before();
    mbar_arrive(bar1);
    if (bar2) mbar_arrive(bar2);
    if (gtile) {
        uint8_t* box = gtile + (v >> 6) * 8192;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            *reinterpret_cast<__nv_bfloat16*>(box + sw128_offset(c0 + i, v & 63)) =
                __float2bfloat16_rn(d0[i]);
        fence_async_smem();
    }
}

// Token row (in the [B*T] token tensors) of chunk n of batch b, and its
// valid rows.  Fixed-length batches: b T + n C and C.  Packed sequences (B =
// 1): the chunk table ctab [NT][2] (first token, valid rows; 0 rows for an
// unused slot).  Only a sequence's last chunk can be partial.
__device__ __forceinline__ int tok_row(const int* ctab, int b, int T, int n) {
    return ctab ? ctab[2 * n] : b * T + n * kC;
}
__device__ __forceinline__ int tok_len(const int* ctab, int n) {
    return ctab ? ctab[2 * n + 1] : kC;
}
// Zeroes rows [len, 64) of a [64][128] bf16 token tile (two 128B-swizzled
// 64-column boxes, 8 KB apart; a row of a box is 128 contiguous bytes).
__device__ __forceinline__ void zero_tile_rows(uint8_t* tile, int len, int tid, int nthreads) {
    const int n16 = (kC - len) * 16;   // 16-byte units: 8 per row and box
    for (int i = tid; i < n16; i += nthreads) {
        const int r = len + (i >> 4), box = (i >> 3) & 1, u = i & 7;
        *reinterpret_cast<uint4*>(tile + box * 8192 + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
    }
}
// Copies a [D][D] fp32 state (zeros if src is null): an empty sequence's
// final state is its initial state, and its dh0 is its dht.
__device__ __forceinline__ void copy_state(float* dst, const float* src, int D, int tid,
                                           int nthreads) {
    for (int e = tid; e < D * D; e += nthreads) dst[e] = src ? src[e] : 0.f;
}

struct ChainArgs {
    int B, T, HV, NT;
    int D;              // K = V of the tensors (64 or 128); the kernel works at 128
    const float* gam;   // [BH*NT][128]
    const float* h0;    // [BH][K][V] or null
    __nv_bfloat16* o;   // [B,T,HV,V]
    float* ht;          // [BH][K][V] or null
    __nv_bfloat16* h_out;  // [BH][NT][V][K] or null (states at chunk starts, transposed, bf16)
    __nv_bfloat16* delta_out;  // [BH][NT][V][C] or null (transposed); set iff h_out is
    // Two-term split of U and delta (the backward with an upstream final-state
    // gradient): U = U2 + u_lo read from [BH*T][128], and the low parts of
    // delta^T to delta_lo ([BH][NT][V][C], like delta_out).  Both or neither.
    const __nv_bfloat16* u_lo;
    __nv_bfloat16* delta_lo;
    // Segmented scan of long sequences (nseg >= 3; 0: one CTA per head over
    // all chunks).  The chunks are cut into nseg segments of seglen (the last
    // may be shorter).  pass 1: CTAs [0, BH) run segment 0 in full (its end
    // state into sbuf[.][1]); CTAs [BH, BH (nseg-1)) run segments 1..nseg-2
    // from zero, their end states into zbuf; CTAs [BH (nseg-1), BH (2 nseg-3))
    // run the same segments from the identity with U = 0, their transition
    // matrices into mbuf.  pass 3: CTAs [0, BH (nseg-1)) run segments
    // 1..nseg-1 in full from sbuf (the last one's end state into ht).
    // Buffers: [BH][nseg][K][V] fp32 at the tensors' width; ident [K][V].
    int nseg, seglen, pass;
    float *sbuf, *zbuf, *mbuf;
    const float* ident;
    // Packed sequences (B = 1; null for fixed-length batches): the chunk
    // table and each sequence's first chunk slot; CTA c runs sequence c / HV
    // of value head c % HV over its chunk slots, with h0 / ht at row c.
    const int *ctab, *sfirst;
};

// The work of one chain CTA: head bh walks chunks n0 .. n0 + cnt - 1 from
// h0 ([D][D], null: zero) with U taken as zero if zero_u, writes o if
// write_o, and its end state to ht ([D][D], null: none).
struct ChainJob {
    int bh, n0, cnt;
    bool write_o, zero_u;
    const float* h0;
    float* ht;
};

template <bool VL>
__device__ __forceinline__ ChainJob chain_job(const ChainArgs& a, int c) {
    const int BH = a.B * a.HV;
    const size_t S = (size_t)a.D * a.D;
    ChainJob j;
    j.zero_u = false;
    if (VL && a.sfirst) {
        const int sq = c / a.HV;
        j.bh = c % a.HV;
        j.n0 = a.sfirst[sq];
        j.cnt = a.sfirst[sq + 1] - j.n0;
        j.write_o = a.o != nullptr;
        j.h0 = a.h0 ? a.h0 + (size_t)c * S : nullptr;
        j.ht = a.ht ? a.ht + (size_t)c * S : nullptr;
        return j;
    }
    if (a.nseg == 0) {
        j.bh = c;
        j.n0 = 0;
        j.cnt = a.NT;
        j.write_o = a.o != nullptr;
        j.h0 = a.h0 ? a.h0 + (size_t)c * S : nullptr;
        j.ht = a.ht ? a.ht + (size_t)c * S : nullptr;
        return j;
    }
    auto seg = [&](int p) {
        j.n0 = p * a.seglen;
        j.cnt = min(a.seglen, a.NT - j.n0);
    };
    auto buf = [&](float* base, int p) { return base + ((size_t)j.bh * a.nseg + p) * S; };
    j.bh = c % BH;
    if (a.pass == 1) {
        const int role = c / BH;   // 0: segment 0; 1..nseg-2: Z; nseg-1..2 nseg-4: M
        if (role == 0) {
            seg(0);
            j.write_o = true;
            j.h0 = a.h0 ? a.h0 + (size_t)j.bh * S : nullptr;
            j.ht = buf(a.sbuf, 1);
        } else if (role <= a.nseg - 2) {
            seg(role);
            j.write_o = false;
            j.h0 = nullptr;
            j.ht = buf(a.zbuf, role);
        } else {
            const int p = role - (a.nseg - 2);
            seg(p);
            j.write_o = false;
            j.zero_u = true;
            j.h0 = a.ident;
            j.ht = buf(a.mbuf, p);
        }
    } else {
        const int p = c / BH + 1;
        seg(p);
        j.write_o = true;
        j.h0 = buf(a.sbuf, p);
        j.ht = p == a.nseg - 1 && a.ht ? a.ht + (size_t)j.bh * S : nullptr;
    }
    return j;
}

// LO: U comes as two parts (a.u_lo added) and delta's low parts go to
// a.delta_lo; a separate instantiation, so that the plain one's serial
// chunk loop carries none of it.
template <bool LO, bool VL>
__global__ void __launch_bounds__(kChainThreads, 1)
chain_fwd_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_kbt,
                 const __grid_constant__ CUtensorMap tm_aqk,
                 const __grid_constant__ CUtensorMap tm_u,
                 const __grid_constant__ CUtensorMap tm_hout,
                 const __grid_constant__ CUtensorMap tm_dout,
                 const __grid_constant__ CUtensorMap tm_o, ChainArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // [2]
    uint64_t* empty = full + 2;                                     // [2]
    uint64_t* bar_S = full + 4;
    uint64_t* bar_delta = full + 5;
    uint64_t* bar_D12 = full + 6;
    uint64_t* bar_D3 = full + 7;
    uint64_t* bar_fin = full + 8;
    uint64_t* bar_Sx = full + 9;   // state rescaled in TMEM
    uint64_t* bar_o = full + 10;   // [2] the epilogue is done with a stage (and its U area)
    uint64_t* bar_u = full + 12;   // every epilogue thread has read its U values
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full + 13);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ChainJob job = chain_job<VL>(a, blockIdx.x);
    const int bh = job.bh;
    const int b = bh / a.HV, hv = bh % a.HV;
    const int NT = job.cnt;      // chunks of this CTA: n0 .. n0 + NT - 1
    const int n0 = job.n0;
    const bool write_o = job.write_o && a.o;

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&empty[0], 1);
        mbar_init(&empty[1], 1);
        mbar_init(bar_S, kChainEpi);
        mbar_init(bar_delta, kChainEpi);
        mbar_init(bar_D12, 1);
        mbar_init(bar_D3, 1);
        mbar_init(bar_fin, 1);
        mbar_init(bar_Sx, kChainEpi);
        mbar_init(&bar_o[0], kChainEpi);
        mbar_init(&bar_o[1], kChainEpi);
        mbar_init(bar_u, kChainEpi);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_kbt);
            prefetch_tmap(&tm_aqk);
            prefetch_tmap(&tm_u);
            // Hands back the stage of epilogue iteration j (its U area then
            // holds the output tile of chunk j - 1, stored here by TMA; its
            // source must be read before the stage is refilled).
            auto drain_o = [&](int j) -> bool {
                const int sj = j & 1;
                if (!wait_bar(&bar_o[sj], (j >> 1) & 1, 21)) return false;
                if (write_o && j >= 1) {
                    const int z = tok_row((VL ? a.ctab : nullptr), b, a.T, n0 + j - 1);
                    const uint8_t* tile = smem + sj * STAGE_BYTES + OFF_U;
                    tma_store_3d(&tm_o, tile, 0, hv, z);
                    if (a.D > 64) tma_store_3d(&tm_o, tile + 8192, 64, hv, z);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
                return true;
            };
            int issued = 0;
            for (int n = 0; n < NT; ++n) {
                const int s = n & 1;
                if (!wait_bar(&empty[s], ((n >> 1) & 1) ^ 1, 1)) break;
                if (n >= 2 && !drain_o(n - 2)) break;
                uint8_t* st = smem + s * STAGE_BYTES;
                // a CTA that writes no output reads neither Qh nor Aqk
                mbar_arrive_expect_tx(&full[s], write_o ? STAGE_TX : STAGE_TX - 16384 - 8192);
                const int row = bh * a.T + (n0 + n) * kC;
                const int crow = bh * a.NT + n0 + n;
                tma_load_2d(st + OFF_W, &tm_w, &full[s], 0, row);
                tma_load_2d(st + OFF_W + 8192, &tm_w, &full[s], 64, row);
                if (write_o) {
                    tma_load_2d(st + OFF_Q, &tm_q, &full[s], 0, row);
                    tma_load_2d(st + OFF_Q + 8192, &tm_q, &full[s], 64, row);
                    tma_load_2d(st + OFF_AQK, &tm_aqk, &full[s], 0, crow * kC);
                }
                tma_load_2d(st + OFF_KBT, &tm_kbt, &full[s], 0, row);
                tma_load_2d(st + OFF_KBT + 8192, &tm_kbt, &full[s], 64, row);
                tma_load_2d(st + OFF_U, &tm_u, &full[s], 0, row);
                bulk_load(smem + OFF_GAM + s * 512, a.gam + (size_t)crow * kD, 512, &full[s]);
                issued = n + 1;
                // the chunk two ahead into L2, so that its stage load (issued
                // once this one is consumed) does not wait on DRAM
                if (n + 2 < NT) {
                    const int row2 = row + 2 * kC, crow2 = crow + 2;
                    tma_prefetch_2d(&tm_w, 0, row2);
                    tma_prefetch_2d(&tm_w, 64, row2);
                    if (write_o) {
                        tma_prefetch_2d(&tm_q, 0, row2);
                        tma_prefetch_2d(&tm_q, 64, row2);
                        tma_prefetch_2d(&tm_aqk, 0, crow2 * kC);
                    }
                    tma_prefetch_2d(&tm_kbt, 0, row2);
                    tma_prefetch_2d(&tm_kbt, 64, row2);
                    tma_prefetch_2d(&tm_u, 0, row2);
                    bulk_prefetch_l2(a.gam + (size_t)crow2 * kD, 512);
                    if (LO) bulk_prefetch_l2(a.u_lo + (size_t)row2 * kD, kC * kD * 2);
                }
            }
            // the epilogue's last two iterations (after an error, skipped)
            for (int j = NT - 2 < 0 ? 0 : NT - 2; issued == NT && j < NT; ++j)
                if (!drain_o(j)) break;
            bulk_wait_all();
            // do not leave copies in flight: wait for the last stages issued
            for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n)
                wait_bar(&full[n & 1], (n >> 1) & 1, 2);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc64 = idesc_bf16_f32(128, 64);
            const uint32_t idesc128 = idesc_bf16_f32(128, 128);
            // descriptors are built once; K offsets are added to the start field
            const uint64_t dS = sdesc_sw128(smem_u32(smem + OFF_S));
            const uint64_t dD = sdesc_sw128(smem_u32(smem + OFF_DELTA));
            const uint32_t st0 = smem_u32(smem);
            const uint64_t dW0 = sdesc_sw128(st0 + OFF_W), dQ0 = sdesc_sw128(st0 + OFF_Q);
            const uint64_t dKb0 = sdesc_mn_sw128(st0 + OFF_KBT, 8192);
            const uint64_t dAq0 = sdesc_sw128(st0 + OFF_AQK);
            for (int n = 0; n < NT; ++n) {
                const int s = n & 1;
                const uint64_t so = s ? (STAGE_BYTES >> 4) : 0;  // stage offset in 16-byte units

                if (!wait_bar(&full[s], (n >> 1) & 1, 3)) break;
                if (!wait_bar(bar_S, n & 1, 4)) break;
                tc_fence_after();
                const uint32_t tO = tmem + ((n & 1) ? TM_O1 : TM_O0);
                const uint64_t dSn = dS + (uint64_t)((n & 1) * (S_TILE >> 4));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ka = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                    const uint32_t kb = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                    mma_bf16(tmem + TM_W, dSn + ka, dW0 + so + kb, idesc64, kk > 0);
                }
                // the delta step rewrites the delta tile once D12 completes: the
                // previous delta's store must have read it
                if (a.h_out) bulk_wait_read_all();
                mma_commit(bar_D12);
                // stores are issued after the products they would otherwise delay
                if (a.h_out) {  // S_n^T tile (rows v) as it stands to h_out, by TMA
                    const int y = (bh * a.NT + n0 + n) * kD;
                    uint8_t* tile = smem + OFF_S + (n & 1) * S_TILE;
                    tma_store_2d(&tm_hout, tile, 0, y);
                    tma_store_2d(&tm_hout, tile + 16384, 64, y);
                    bulk_commit_group();
                }
                if (!wait_bar(bar_delta, n & 1, 5)) break;
                tc_fence_after();
                if (!wait_bar(bar_Sx, n & 1, 10)) break;  // S^T rescaled by gam in TMEM
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // Kb tile [64 c][128 k] read MN-major (N = k)
                    mma_bf16(tmem + TM_S, dD + ((kk * 32) >> 4), dKb0 + so + ((kk * 2048) >> 4),
                             idesc128 | kBMajorMN, 1);
                // the next state step may start once the state update is done
                // and the previous chunk's state store (groups: its state,
                // its delta, this chunk's state) has read the tile it will
                // rewrite; O_n is read only after the next chunk's D12, which
                // also covers it
                if (a.h_out) bulk_wait_read_but2();
                mma_commit(bar_D3);
                // O_n = Qh S_n + Aqk delta (rows t in TMEM lanes 0..63, columns
                // v), behind the state update (the S tile of parity n is
                // rewritten only after the next D3).  A = the Qh and Aqk tiles
                // with M = 128: their rows 64..127 are the next 64 rows of the
                // stage, don't-care; B = the S^T and delta^T tiles (N = v).
                if (write_o) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ka = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        const uint32_t kb = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                        mma_bf16(tO, dQ0 + so + kb, dSn + ka, idesc128, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tO, dAq0 + so + ((kk * 32) >> 4), dD + ((kk * 32) >> 4), idesc128,
                                 1);
                }
                mma_commit(&empty[s]);
                if (a.delta_out) {  // delta_n^T tile (rows v) to delta_out, by TMA
                    tma_store_2d(&tm_dout, smem + OFF_DELTA, 0, (bh * a.NT + n0 + n) * kD);
                    bulk_commit_group();
                }
            }
            bulk_wait_all();
            // all issued MMAs complete before TMEM is released
            mma_commit(bar_fin);
            wait_bar(bar_fin, 0, 6);
        }
    } else {
        // ---------------- epilogue: thread <-> value column v ----------------
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int v = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint8_t* sDelta = smem + OFF_DELTA;
        float r[32];
        bool ok = true;

        // E1: S_n -> bf16 operand tile (of parity n); then, once chunk n's
        // stage (gam) has landed, the TMEM copy scaled by gam_n.
        auto e1 = [&](int n) -> bool {
            const int s = n & 1;
            float r0[32], r1[32];
            chain_state_tile(tmem + lane_off + TM_S, smem + OFF_S + s * S_TILE, n == 0, job.h0,
                             a.D, v, half, bar_S, r0, r1);
            if (!wait_bar_warp(&full[s], (n >> 1) & 1, 7)) return false;
            chain_state_rescale(tmem + lane_off + TM_S,
                                reinterpret_cast<const float*>(smem + OFF_GAM + s * 512), half,
                                bar_Sx, r0, r1);
            return true;
        };

        // E3: output rows of chunk m (row t = TMEM lane, warps of lanes 0..63;
        // thread (t, half) holds columns v in [64 half, 64 half + 64)) into a
        // 128B-swizzled pair of [64 t][64 v] tiles at dst, or, for the last
        // chunk, straight to global memory
        auto o_rows = [&](int m, float (&x0)[32], float (&x1)[32]) {
            const uint32_t tO = (m & 1) ? TM_O1 : TM_O0;
            tmem_ld32_nw(tmem + lane_off + tO + half * 64, x0);
            tmem_ld32_nw(tmem + lane_off + tO + half * 64 + 32, x1);
            tmem_wait_ld_dep(x0);
            tmem_wait_ld_dep(x1);
        };
        auto o_tile = [&](int m, uint8_t* dst) {
            if (q >= 2) return;
            float x1[32];
            o_rows(m, r, x1);
            uint8_t* box = dst + half * 8192;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float e0[8], e1v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    e0[i] = r[8 * j + i];
                    e1v[i] = x1[8 * j + i];
                }
                *reinterpret_cast<uint4*>(box + sw128_offset(v, 8 * j)) = pack8(e0);
                *reinterpret_cast<uint4*>(box + sw128_offset(v, 32 + 8 * j)) = pack8(e1v);
            }
        };
        auto o_out = [&](int m) {
            if (q >= 2 || half * 64 >= a.D) return;   // warp-uniform: the TMEM load is .aligned
            float x1[32];
            o_rows(m, r, x1);
            // rows past a partial chunk's end belong to the next sequence
            if (v >= tok_len((VL ? a.ctab : nullptr), n0 + m)) return;
            __nv_bfloat16* op =
                a.o + (((size_t)tok_row((VL ? a.ctab : nullptr), b, a.T, n0 + m) + v) * a.HV + hv) * a.D + half * 64;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float e0[8], e1v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    e0[i] = r[8 * j + i];
                    e1v[i] = x1[8 * j + i];
                }
                *reinterpret_cast<uint4*>(op + 8 * j) = pack8(e0);
                *reinterpret_cast<uint4*>(op + 32 + 8 * j) = pack8(e1v);
            }
        };

        if (NT == 0) {   // an empty sequence: ht = h0
            if (job.ht) copy_state(job.ht, job.h0, a.D, threadIdx.x - 64, kChainEpi);
            ok = false;
        } else {
            ok = e1(0);
        }
        for (int n = 0; ok && n < NT; ++n) {
            const int s = n & 1;
            // E2: delta^T = U^T - S^T W^T  -> bf16 operand tile.  U (in the
            // stage since E1 of this chunk) is read while the products run.
            float u[32];
            {
                const __nv_bfloat16* U =
                    reinterpret_cast<const __nv_bfloat16*>(smem + s * STAGE_BYTES + OFF_U);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    u[i] = job.zero_u ? 0.f : __bfloat162float(U[(32 * half + i) * kD + v]);
                if (LO && !job.zero_u) {
                    const __nv_bfloat16* ul =
                        a.u_lo + ((size_t)bh * a.T + (size_t)(n0 + n) * kC + 32 * half) * kD + v;
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] += __bfloat162float(ul[(size_t)i * kD]);
                }
            }
            if (!wait_bar_warp(bar_D12, n & 1, 8)) { ok = false; break; }
            tc_fence_after();
            chain_delta_step(
                tmem + lane_off + TM_W, sDelta, u, false, v, half, bar_delta, nullptr, nullptr,
                LO ? a.delta_lo + (((size_t)bh * a.NT + n0 + n) * kD + v) * kC + 32 * half
                   : nullptr);
            // the previous chunk's output, while this chunk's state update
            // runs, into the U area of this chunk's stage once every thread
            // has read its U values; the TMA thread stores it
            if (write_o) {
                mbar_arrive(bar_u);
                if (!wait_bar_warp(bar_u, n & 1, 22)) { ok = false; break; }
                if (n > 0) o_tile(n - 1, smem + s * STAGE_BYTES + OFF_U);
                fence_async_smem();
            }
            mbar_arrive(&bar_o[s]);
            if (!wait_bar_warp(bar_D3, n & 1, 9)) { ok = false; break; }
            tc_fence_after();
            if (n + 1 < NT) {
                if (!e1(n + 1)) { ok = false; break; }
            } else if (job.ht) {
#pragma unroll 1
                for (int cb = 2 * half; cb < 2 * half + 2; ++cb) {
                    tmem_ld32(tmem + lane_off + TM_S + cb * 32, r);
                    if (v >= a.D || cb * 32 >= a.D) continue;   // [D][D]
                    float* hp = job.ht + (size_t)(cb * 32) * a.D + v;
#pragma unroll
                    for (int i = 0; i < 32; ++i) hp[(size_t)i * a.D] = r[i];
                }
            }
        }
        // the last chunk's output products are covered by the final commit only
        if (ok && write_o && wait_bar_warp(bar_fin, 0, 6)) {
            tc_fence_after();
            o_out(NT - 1);
        }
        (void)ok;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// Combine step of the segmented scan: per head, the true start state of
// segment p + 1 is M_p S_p + Z_p for p = 1 .. nseg - 2 (S_1 comes from the
// full run of segment 0).  One CTA of 256 threads per head; thread (j, h)
// owns column j and rows 64 h .. 64 h + 63 of the [D][D] result (D <= 128),
// so that a warp's global loads of Z and stores of the result cover 128
// contiguous bytes of a row.  M is held transposed in shared memory with a
// row stride of D + 4 floats: a thread's 64 rows at one k are 16 broadcast
// float4 loads, and S_p[k][j] one conflict-free load.
__global__ void __launch_bounds__(256)
chain_combine_kernel(int D, int nseg, float* __restrict__ sbuf, const float* __restrict__ zbuf,
                     const float* __restrict__ mbuf) {
    extern __shared__ float cs[];
    const int MT = D + 4;
    float* Mt = cs;                  // Mt[k * MT + i] = M[i][k]; MT * 4 bytes is 16-byte aligned
    float* Sk = cs + D * MT;         // S[k][j]
    const int bh = blockIdx.x, tid = threadIdx.x;
    const size_t SZ = (size_t)D * D;
    const int j = tid & 127, i0 = (tid >> 7) * 64;
    for (int p = 1; p <= nseg - 2; ++p) {
        const float* M = mbuf + ((size_t)bh * nseg + p) * SZ;
        const float* Sp = sbuf + ((size_t)bh * nseg + p) * SZ;
        __syncthreads();   // the previous step's rows are written
        // 16-byte loads (D is a multiple of 4; the buffers are 16-byte aligned)
        for (int e4 = tid; e4 < D * D / 4; e4 += 256) {
            const float4 m = reinterpret_cast<const float4*>(M)[e4];
            const int i = (4 * e4) / D, k = (4 * e4) % D;
            Mt[k * MT + i] = m.x;
            Mt[(k + 1) * MT + i] = m.y;
            Mt[(k + 2) * MT + i] = m.z;
            Mt[(k + 3) * MT + i] = m.w;
            reinterpret_cast<float4*>(Sk)[e4] = reinterpret_cast<const float4*>(Sp)[e4];
        }
        __syncthreads();
        if (j < D && i0 < D) {
            float acc[64];
            const float* Z = zbuf + ((size_t)bh * nseg + p) * SZ + (size_t)i0 * D + j;
#pragma unroll
            for (int ii = 0; ii < 64; ++ii) acc[ii] = Z[(size_t)ii * D];
            for (int k = 0; k < D; ++k) {
                const float sv = Sk[k * D + j];
                const float4* mrow = reinterpret_cast<const float4*>(Mt + k * MT + i0);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 m = mrow[q];
                    acc[4 * q] = fmaf(m.x, sv, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(m.y, sv, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(m.z, sv, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(m.w, sv, acc[4 * q + 3]);
                }
            }
            float* out = sbuf + ((size_t)bh * nseg + p + 1) * SZ + (size_t)i0 * D + j;
#pragma unroll
            for (int ii = 0; ii < 64; ++ii) out[(size_t)ii * D] = acc[ii];
        }
    }
}

// The D x D identity (the start of the transition runs of the segmented scan).
__global__ void fill_identity_kernel(float* __restrict__ I, int D) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < D * D; e += gridDim.x * blockDim.x)
        I[e] = (e / D == e % D) ? 1.f : 0.f;
}

// ===========================================================================
// Reverse state pass (backward chain).  One CTA per (b, hv) walks the chunks
// from last to first with dS (gradient of the state at the END of the
// current chunk) on chip, fp32 in TMEM, transposed (lane = value column):
//     ddelta^T = dS^T Kb^T + dO^T Aqk                 (M=128 v, N=64 rows)
//     dS0^T    = diag(gam) dS^T + dO^T Qh - ddelta^T W   (M=128 v, N=128 k)
// dO, Aqk, Qh and W are used straight from their TMA tiles as MN-major
// operands; dS^T and -ddelta^T are written by the epilogue as K-major tiles.
// Writes dS of every chunk (bf16 [K][V]) and ddelta (bf16 [C][V]) for the
// gradient kernel, and dh0.
// ===========================================================================
constexpr uint32_t RB_DO = 0;        // dO [64 t][128 v]: two 64-column boxes, 8 KB apart
constexpr uint32_t RB_Q = 16384;     // Qh [64 t][128 k]
constexpr uint32_t RB_W = 32768;     // W  [64 r][128 k]
constexpr uint32_t RB_KBT = 49152;   // Kb [64 r][128 k]
constexpr uint32_t RB_AQK = 65536;   // Aqk [64 t][64 r]
constexpr uint32_t TM2_S = 0, TM2_DD = 128, TM2_COLS = 256;

struct ChainBwdArgs {
    int B, T, HV, NT;
    const int *ctab, *sfirst;    // packed sequences (as in ChainArgs), or null
    int D;              // K = V of the tensors (64 or 128); the kernel works at 128
    const float* gam;
    const float* dht;            // [BH][K][V] or null
    float* dh0;                  // [BH][K][V] or null
    __nv_bfloat16* dh_out;       // [BH][NT][V][K] (transposed)
    __nv_bfloat16* dh_lo;        // low parts of dh_out (x - bf16(x)), same layout, or null
};

// LO: also write the low parts of dS (a.dh_lo); a separate instantiation,
// so that the plain one keeps its registers.
template <bool LO, bool VL>
__global__ void __launch_bounds__(kChainThreads, 1)
chain_bwd_kernel(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_kbt,
                 const __grid_constant__ CUtensorMap tm_aqk,
                 const __grid_constant__ CUtensorMap tm_dhout,
                 const __grid_constant__ CUtensorMap tm_dd, ChainBwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* empty = full + 2;
    uint64_t* bar_S = full + 4;
    uint64_t* bar_delta = full + 5;
    uint64_t* bar_dd = full + 6;
    uint64_t* bar_D4 = full + 7;
    uint64_t* bar_fin = full + 8;
    uint64_t* bar_Sx = full + 9;   // state rescaled in TMEM
    uint64_t* bar_o = full + 10;   // [2] the epilogue is done with a stage (ddelta tile in it)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's chunk slots n0 .. n0 + NT - 1 of workspace head row bh,
    // walked in reverse; dht and dh0 at state row srow
    int bh, b, hv, n0, NT, srow;
    if ((VL ? a.sfirst : nullptr)) {
        const int sq = blockIdx.x / a.HV;
        hv = blockIdx.x % a.HV;
        bh = hv;
        b = 0;
        n0 = (VL ? a.sfirst : nullptr)[sq];
        NT = (VL ? a.sfirst : nullptr)[sq + 1] - n0;
        srow = blockIdx.x;
    } else {
        bh = blockIdx.x;
        b = bh / a.HV;
        hv = bh % a.HV;
        n0 = 0;
        NT = a.NT;
        srow = bh;
    }

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&empty[0], 1);
        mbar_init(&empty[1], 1);
        mbar_init(bar_S, kChainEpi);
        mbar_init(bar_delta, kChainEpi);
        mbar_init(bar_dd, 1);
        mbar_init(bar_D4, 1);
        mbar_init(bar_fin, 1);
        mbar_init(bar_Sx, kChainEpi);
        mbar_init(&bar_o[0], kChainEpi);
        mbar_init(&bar_o[1], kChainEpi);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TM2_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_kbt);
            prefetch_tmap(&tm_aqk);
            // Hands back the stage of epilogue iteration j: its Kb area (free
            // once ddelta's products completed) then holds ddelta of chunk
            // NT-1-j, stored here by TMA before the stage is refilled.
            auto drain_dd = [&](int j) -> bool {
                const int sj = j & 1;
                if (!wait_bar(&bar_o[sj], (j >> 1) & 1, 23)) return false;
                const int y = bh * a.T + (n0 + NT - 1 - j) * kC;
                const uint8_t* tile = smem + sj * STAGE_BYTES + RB_KBT;
                tma_store_2d(&tm_dd, tile, 0, y);
                tma_store_2d(&tm_dd, tile + 8192, 64, y);
                bulk_commit_group();
                bulk_wait_read_all();
                return true;
            };
            int issued = 0;
            for (int i = 0; i < NT; ++i) {
                const int n = NT - 1 - i, s = i & 1;
                if (!wait_bar(&empty[s], ((i >> 1) & 1) ^ 1, 11)) break;
                if (i >= 2 && !drain_dd(i - 2)) break;
                uint8_t* st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], STAGE_TX);
                const int row = bh * a.T + (n0 + n) * kC;
                const int crow = bh * a.NT + n0 + n;
                const int trow = tok_row((VL ? a.ctab : nullptr), b, a.T, n0 + n);
                tma_load_3d(st + RB_DO, &tm_do, &full[s], 0, hv, trow);
                tma_load_3d(st + RB_DO + 8192, &tm_do, &full[s], 64, hv, trow);
                tma_load_2d(st + RB_Q, &tm_q, &full[s], 0, row);
                tma_load_2d(st + RB_Q + 8192, &tm_q, &full[s], 64, row);
                tma_load_2d(st + RB_W, &tm_w, &full[s], 0, row);
                tma_load_2d(st + RB_W + 8192, &tm_w, &full[s], 64, row);
                tma_load_2d(st + RB_KBT, &tm_kbt, &full[s], 0, row);
                tma_load_2d(st + RB_KBT + 8192, &tm_kbt, &full[s], 64, row);
                tma_load_2d(st + RB_AQK, &tm_aqk, &full[s], 0, crow * kC);
                bulk_load(smem + OFF_GAM + s * 512, a.gam + (size_t)crow * kD, 512, &full[s]);
                issued = i + 1;
                // the chunk two ahead (n - 2) into L2
                if (n >= 2) {
                    const int row2 = row - 2 * kC, crow2 = crow - 2;
                    const int trow2 = tok_row((VL ? a.ctab : nullptr), b, a.T, n0 + n - 2);
                    tma_prefetch_3d(&tm_do, 0, hv, trow2);
                    if (a.D > 64) tma_prefetch_3d(&tm_do, 64, hv, trow2);
                    tma_prefetch_2d(&tm_q, 0, row2);
                    tma_prefetch_2d(&tm_q, 64, row2);
                    tma_prefetch_2d(&tm_w, 0, row2);
                    tma_prefetch_2d(&tm_w, 64, row2);
                    tma_prefetch_2d(&tm_kbt, 0, row2);
                    tma_prefetch_2d(&tm_kbt, 64, row2);
                    tma_prefetch_2d(&tm_aqk, 0, crow2 * kC);
                    bulk_prefetch_l2(a.gam + (size_t)crow2 * kD, 512);
                }
            }
            // the epilogue's last two iterations (after an error, skipped)
            for (int j = NT - 2 < 0 ? 0 : NT - 2; issued == NT && j < NT; ++j)
                if (!drain_dd(j)) break;
            bulk_wait_all();
            for (int i = issued - 2 < 0 ? 0 : issued - 2; i < issued; ++i)
                wait_bar(&full[i & 1], (i >> 1) & 1, 12);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id64 = idesc_bf16_f32(128, 64), id128 = idesc_bf16_f32(128, 128);
            const uint64_t dS = sdesc_sw128(smem_u32(smem + OFF_S));
            const uint64_t dD = sdesc_sw128(smem_u32(smem + OFF_DELTA));
            const uint32_t st0 = smem_u32(smem);
            const uint64_t dKb0 = sdesc_sw128(st0 + RB_KBT);
            const uint64_t dDO0 = sdesc_mn_sw128(st0 + RB_DO, 8192);
            const uint64_t dAq0 = sdesc_mn_sw128(st0 + RB_AQK, 8192);
            const uint64_t dQ0 = sdesc_mn_sw128(st0 + RB_Q, 8192);
            const uint64_t dW0 = sdesc_mn_sw128(st0 + RB_W, 8192);
            for (int i = 0; i < NT; ++i) {
                const int s = i & 1;
                const uint64_t so = s ? (STAGE_BYTES >> 4) : 0;  // stage offset in 16-byte units
                if (!wait_bar(&full[s], (i >> 1) & 1, 13)) break;
                if (!wait_bar(bar_S, i & 1, 14)) break;
                tc_fence_after();
                const uint64_t dSi = dS + (uint64_t)((i & 1) * (S_TILE >> 4));
                {  // dS^T tile (rows v, parity i) of chunk n = NT-1-i to dh_out, by TMA
                    const int y = (bh * a.NT + n0 + (NT - 1 - i)) * kD;
                    uint8_t* tile = smem + OFF_S + (i & 1) * S_TILE;
                    tma_store_2d(&tm_dhout, tile, 0, y);
                    tma_store_2d(&tm_dhout, tile + 16384, 64, y);
                    bulk_commit_group();
                }
                // ddelta^T = dS^T Kb^T  (B = Kb tile [64 r][128 k], K-major)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM2_DD, dSi + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                             dKb0 + so + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), id64, kk > 0);
                // ddelta^T += dO^T Aqk
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM2_DD, dDO0 + so + ((kk * 2048) >> 4),
                             dAq0 + so + ((kk * 2048) >> 4), id64 | kAMajorMN | kBMajorMN, 1);
                mma_commit(bar_dd);
                if (!wait_bar(bar_Sx, i & 1, 20)) break;  // dS^T rescaled by gam in TMEM
                tc_fence_after();
                // dS^T += dO^T Qh
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM2_S, dDO0 + so + ((kk * 2048) >> 4),
                             dQ0 + so + ((kk * 2048) >> 4), id128 | kAMajorMN | kBMajorMN, 1);
                if (!wait_bar(bar_delta, i & 1, 15)) break;
                tc_fence_after();
                // dS^T += (-ddelta^T) W
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM2_S, dD + ((kk * 32) >> 4), dW0 + so + ((kk * 2048) >> 4),
                             id128 | kBMajorMN, 1);
                // the next state step rewrites the tile of the previous chunk's
                // store: all but this chunk's store have read their tiles
                bulk_wait_read_but1();
                mma_commit(bar_D4);
                mma_commit(&empty[s]);
            }
            bulk_wait_all();
            mma_commit(bar_fin);
            wait_bar(bar_fin, 0, 16);
        }
    } else {
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int v = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint8_t* sDelta = smem + OFF_DELTA;
        float r[32];
        bool ok = true;

        // E1: dS (end of chunk n) -> bf16 operand tile (of parity i); then,
        // once the chunk's stage (gam) has landed, the TMEM copy scaled by gam_n.
        auto e1 = [&](int i) -> bool {
            const int s = i & 1;
            float r0[32], r1[32];
            chain_state_tile(tmem + lane_off + TM2_S, smem + OFF_S + s * S_TILE, i == 0,
                             a.dht ? a.dht + (size_t)srow * a.D * a.D : nullptr, a.D, v, half, bar_S,
                             r0, r1);
            if (LO) {
                __nv_bfloat16* lo =
                    a.dh_lo + (((size_t)bh * a.NT + n0 + (NT - 1 - i)) * kD + v) * kD + 64 * half;
                store_lo32(lo, r0);
                store_lo32(lo + 32, r1);
            }
            if (!wait_bar_warp(&full[s], (i >> 1) & 1, 17)) return false;
            chain_state_rescale(tmem + lane_off + TM2_S,
                                reinterpret_cast<const float*>(smem + OFF_GAM + s * 512), half,
                                bar_Sx, r0, r1);
            return true;
        };

        if (NT == 0) {   // an empty sequence: dh0 = dht
            if (a.dh0)
                copy_state(a.dh0 + (size_t)srow * a.D * a.D,
                           a.dht ? a.dht + (size_t)srow * a.D * a.D : nullptr, a.D,
                           threadIdx.x - 64, kChainEpi);
            ok = false;
        } else {
            ok = e1(0);
        }
        for (int i = 0; ok && i < NT; ++i) {
            const int s = i & 1;
            if (!wait_bar_warp(bar_dd, i & 1, 18)) { ok = false; break; }
            tc_fence_after();
            // -ddelta^T to the operand tile; ddelta (true sign) into the
            // stage's Kb area, which the TMA thread stores
            chain_delta_step(tmem + lane_off + TM2_DD, sDelta, nullptr, true, v, half, bar_delta,
                             nullptr, smem + s * STAGE_BYTES + RB_KBT);
            mbar_arrive(&bar_o[s]);
            if (!wait_bar_warp(bar_D4, i & 1, 19)) { ok = false; break; }
            tc_fence_after();
            if (i + 1 < NT) {
                if (!e1(i + 1)) { ok = false; break; }
            } else if (a.dh0) {
#pragma unroll 1
                for (int cb = 2 * half; cb < 2 * half + 2; ++cb) {
                    tmem_ld32(tmem + lane_off + TM2_S + cb * 32, r);
                    if (v >= a.D || cb * 32 >= a.D) continue;   // [D][D]
                    float* hp = a.dh0 + ((size_t)srow * a.D + cb * 32) * a.D + v;
#pragma unroll
                    for (int j = 0; j < 32; ++j) hp[(size_t)j * a.D] = r[j];
                }
            }
        }
        (void)ok;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM2_COLS);
}

// ===========================================================================
// Backward contractions over V, per (chunk, head): persistent CTAs, one per
// SM, walk the chunks.  S0 (state at the chunk start) and dS (gradient at its
// end) come from the two chains:
//     D1 = S0 dO^T       = dQh^T      (M=128 k, N=64)
//     D2 = S0 ddelta^T   = -dW^T
//     D3 = dS delta^T    = dKb^T
//     D4 = [dO; ddelta] [delta; v]^T : top-left = dO delta^T (-> dAqk),
//                                      bottom-right = ddelta v^T (-> dTv)
//     D5 = ddelta^T T    = d(beta v)^T (M=128 v, N=64): dv = beta * D5^T,
//                                       dbeta += sum_v D5^T o v
// plus dgam = rowsum(dS o S0).  Results go to the workspace arrays read by
// the chunk-local backward kernel (dQh and dKb through staging tiles and one
// TMA store each); dv is written directly.
// ===========================================================================
constexpr uint32_t G_S0 = 0, G_DS = 32768, G_ODD = 65536, G_DV = 98304, G_T = 131072;
// v tiles, double-buffered: buffer b's two 64-column boxes at G_DV + vbuf(b)
// and 16 KB later (the stride of the [dO; ddelta] k-blocks its product reads)
__host__ __device__ constexpr uint32_t vbuf(int b) { return b ? 0u : 8192u; }
constexpr uint32_t G_DT = 139264;  // delta^T [128 v][64 c], 16 KB
constexpr uint32_t G_BAR = G_DT + 16384, G_DBV = G_BAR + 64;
// dQh and dKb staged, fp32 [64 rows][128 k] row-major, for one TMA store each
constexpr uint32_t G_STQ = (G_DBV + 2304 + 1023) & ~1023u, G_STK = G_STQ + 32768;
constexpr uint32_t GRAD_TX = 4 * 32768 + 8192;
constexpr uint32_t GRAD_SMEM = G_STK + 32768 + 1024;
static_assert(GRAD_SMEM <= 232448, "grad_v exceeds the per-CTA shared memory limit");
// 8 warps (two per SM sub-partition, so up to 255 registers a thread): thread
// 0 issues the TMA copies and the MMAs, then all eight run the epilogue
constexpr int kGradThreads = 256;

struct GradArgs {
    int T, HV, NT, BH;
    int D;              // V of the tensors (64 or 128); the kernel works at 128
    const __nv_bfloat16* beta;  // [B,T,HV]
    __nv_bfloat16* dv;          // [B,T,HV,V]
    float *dQh, *dKb, *dgam, *dTv, *dbv;
    __nv_bfloat16 *dW, *dAqk;  // bf16: the local backward uses them only as MMA operands
    const int* ctab;           // packed sequences: the chunk table, or null
};

// DW: V of the tensors (64 or 128), a compile-time constant so that the
// 128-wide instantiation indexes exactly as a kernel written for 128 does.
template <int DW, bool VL>
__global__ void __launch_bounds__(kGradThreads, 1)
grad_v_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_dh,
              const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dd,
              const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_t, const __grid_constant__ CUtensorMap tm_dqh,
              const __grid_constant__ CUtensorMap tm_dkb, GradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + G_BAR);   // all tiles but v
    uint64_t* bar_mma = bar_tma + 1;
    uint64_t* bar_v = bar_tma + 2;                                     // v tile, buffer 0
    uint64_t* bar_sd = bar_tma + 3;    // S0 and dS tiles
    uint64_t* bar_s = bar_tma + 4;     // the products that read S0 and dS are done
    uint64_t* bar_dg = bar_tma + 5;    // every thread is done reading S0 and dS
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_tma + 6);
    uint64_t* bar_v1 = bar_tma + 7;                                    // v tile, buffer 1
    float* dbv_part = reinterpret_cast<float*>(smem + G_DBV);  // [4 lane quadrants][64]
    float* beta_s = dbv_part + 4 * 64;                          // [64]
    float* dg_part = beta_s + 64;                               // [2 halves][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = a.NT, total = a.BH * NT;   // CTA i takes chunks i, i + grid, ...

    // thread 0's counts of issued and consumed loads (every load is waited for
    // before the CTA exits)
    int main_issued = 0, v_issued = 0, main_waited = 0, v_waited = 0;
    int sd_issued = 0, sd_waited = 0;
    auto issue_sd = [&](int ch) {     // states, state gradients
        mbar_arrive_expect_tx(bar_sd, 65536);
        tma_load_2d(smem + G_S0, &tm_h, bar_sd, 0, ch * kD);
        tma_load_2d(smem + G_S0 + 16384, &tm_h, bar_sd, 64, ch * kD);
        tma_load_2d(smem + G_DS, &tm_dh, bar_sd, 0, ch * kD);
        tma_load_2d(smem + G_DS + 16384, &tm_dh, bar_sd, 64, ch * kD);
        ++sd_issued;
    };
    auto issue_main = [&](int ch) {   // [dO; ddelta], delta^T, T
        const int nn = ch % NT, bb = ch / NT, hvv = bb % a.HV;
        const int rw = bb * a.T + nn * kC, tr = tok_row((VL ? a.ctab : nullptr), bb / a.HV, a.T, nn);
        mbar_arrive_expect_tx(bar_tma, GRAD_TX - 16384 - 65536);
        tma_load_3d(smem + G_ODD, &tm_do, bar_tma, 0, hvv, tr);
        tma_load_3d(smem + G_ODD + 16384, &tm_do, bar_tma, 64, hvv, tr);
        tma_load_2d(smem + G_ODD + 8192, &tm_dd, bar_tma, 0, rw);
        tma_load_2d(smem + G_ODD + 24576, &tm_dd, bar_tma, 64, rw);
        tma_load_2d(smem + G_DT, &tm_d, bar_tma, 0, ch * kD);
        tma_load_2d(smem + G_T, &tm_t, bar_tma, 0, ch * kC);
        ++main_issued;
    };
    // the i-th v load of the CTA (chunk blockIdx.x + i grid) goes to buffer
    // i & 1 and completes phase (i >> 1) & 1 of that buffer's barrier
    auto issue_v = [&](int ch) {
        const int nn = ch % NT, bb = ch / NT, hvv = bb % a.HV;
        const int tr = tok_row((VL ? a.ctab : nullptr), bb / a.HV, a.T, nn);
        const int b = v_issued & 1;
        uint64_t* bar = b ? bar_v1 : bar_v;
        mbar_arrive_expect_tx(bar, 16384);
        tma_load_3d(smem + G_DV + vbuf(b), &tm_v, bar, 0, hvv, tr);
        tma_load_3d(smem + G_DV + vbuf(b) + 16384, &tm_v, bar, 64, hvv, tr);
        ++v_issued;
    };
    auto load_beta = [&](int ch) {
        const int nn = ch % NT, bb = ch / NT;
        return tid < tok_len((VL ? a.ctab : nullptr), nn)   // 0 past a packed sequence's end
                   ? __bfloat162float(a.beta[((size_t)tok_row((VL ? a.ctab : nullptr), bb / a.HV, a.T, nn) + tid) *
                                                 a.HV + bb % a.HV])
                   : 0.f;
    };

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_v1, 1);
        mbar_init(bar_sd, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_dg, kGradThreads);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (tid == 0 && (int)blockIdx.x < total) {
        issue_sd(blockIdx.x);
        issue_main(blockIdx.x);
        issue_v(blockIdx.x);
        if ((int)(blockIdx.x + gridDim.x) < total) issue_v(blockIdx.x + gridDim.x);
    }
    float beta_next = (tid < kC && (int)blockIdx.x < total) ? load_beta(blockIdx.x) : 0.f;
    bool ok = true;

#pragma unroll 1
    for (int it = 0, chunk = blockIdx.x; chunk < total; ++it, chunk += gridDim.x) {
        const uint32_t ph = it & 1;
        const int next = chunk + gridDim.x;
        const int n = chunk % NT, bh = chunk / NT;
        const int b = bh / a.HV, hv = bh % a.HV;
        const int row = bh * a.T + n * kC;
        const int crow = chunk;
        const int trow = tok_row((VL ? a.ctab : nullptr), b, a.T, n);
        const int len = tok_len((VL ? a.ctab : nullptr), n);   // rows past it belong to the next sequence
        if (tid < kC) {
            beta_s[tid] = beta_next;                          // read after later barriers
            if (next < total) beta_next = load_beta(next);    // in flight meanwhile
        }
        if (tid == 0) {   // the thread that issues the loads also issues the products
            if (wait_bar(bar_sd, ph, 26) && wait_bar(bar_tma, ph, 21) &&
                wait_bar((it & 1) ? bar_v1 : bar_v, (it >> 1) & 1, 25)) {
                ++sd_waited;
                ++main_waited;
                ++v_waited;
                tc_fence_after();
                const uint32_t id64 = idesc_bf16_f32(128, 64), id128 = idesc_bf16_f32(128, 128);
                const uint32_t s0 = smem_u32(smem + G_S0), ds = smem_u32(smem + G_DS);
                const uint32_t odd = smem_u32(smem + G_ODD),
                               dvt = smem_u32(smem + G_DV + vbuf(it & 1));
                const uint32_t tt = smem_u32(smem + G_T), dt = smem_u32(smem + G_DT);
                // the products that read S0 and dS first, so that their tiles
                // can be refilled while the others run
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    // S0 and dS are stored transposed (rows v): A operands read
                    // MN-major, K = v advancing 16 rows per step
                    const uint64_t as0 = sdesc_mn_sw128(s0 + kk * 2048, 16384);
                    const uint64_t ads = sdesc_mn_sw128(ds + kk * 2048, 16384);
                    // S0 [dO; ddelta]^T in one N = 128 product: D1 (dQh^T) columns
                    // 0-63, D2 (dW^T) columns 64-127
                    mma_bf16(tmem + 0, as0, sdesc_sw128(odd + ko), id128 | kAMajorMN, kk > 0);
                    // delta is stored transposed (rows v): B operand read MN-major
                    const uint64_t bdt = sdesc_mn_sw128(dt + kk * 2048, 16384);
                    mma_bf16(tmem + 128, ads, bdt, id64 | kAMajorMN | kBMajorMN, kk > 0);
                }
                mma_commit(bar_s);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t bdt = sdesc_mn_sw128(dt + kk * 2048, 16384);
                    mma_bf16(tmem + 256, sdesc_sw128(odd + ko), bdt, id64 | kBMajorMN, kk > 0);
                    mma_bf16(tmem + 320, sdesc_sw128(odd + ko), sdesc_sw128(dvt + ko), id64,
                             kk > 0);
                }
                // D5 = ddelta^T T: ddelta tile read MN-major (v blocks 16 KB apart), T MN-major
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + 192, sdesc_mn_sw128(odd + 8192 + kk * 2048, 16384),
                             sdesc_mn_sw128(tt + kk * 2048, 8192), id64 | kAMajorMN | kBMajorMN,
                             kk > 0);
                mma_commit(bar_mma);
            }
        }
        __syncwarp();
        // all 8 warps, two per TMEM lane quadrant, splitting the columns
        const int q = warp & 3, half = warp >> 2;
        const int l = q * 32 + lane;  // TMEM lane: k for D1-D3, row for D4, v for D5
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        float r[32];
        ok = ok && wait_bar_warp(bar_sd, ph, 23);
        // dgam[k] = sum_v dS[v][k] S0[v][k] from the bf16 tiles (independent of
        // the MMAs); thread (k = l, half) sums rows v in [64 half, 64 half + 64)
        {
            float acc = 0.f;
            if (ok) {
                const uint32_t kb = (l >> 6) * 16384;
#pragma unroll 8
                for (int vv = 0; vv < 64; ++vv) {
                    const uint32_t off = kb + sw128_offset(64 * half + vv, l & 63);
                    acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + G_S0 + off)) *
                           __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + G_DS + off));
                }
            }
            dg_part[half * kD + l] = acc;
        }
        // S0 and dS are free once every thread has read them and their
        // products are done: the next chunk's copies start now
        fence_async_smem();
        mbar_arrive(bar_dg);
        if (tid == 0 && ok && next < total) {
            if (wait_bar(bar_s, ph, 27) && wait_bar(bar_dg, ph, 28))
                issue_sd(next);
            else
                ok = false;
        }
        ok = ok && wait_bar_warp(bar_mma, ph, 24);
        // [dO; ddelta], delta^T and T are read only by the products, which are
        // done: the next chunk's copies of them start while this chunk's
        // results leave
        if (tid == 0 && ok && next < total) issue_main(next);
        // the previous chunk's dQh / dKb stores have read their staging tiles
        if (tid == 0) bulk_wait_read_all();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (ok) {
            const size_t rb = (size_t)row * kD;
            const int cb = half;  // columns 32*cb .. 32*cb+31 of D1-D3 and D5
            float* stq = reinterpret_cast<float*>(smem + G_STQ);
            float* stk = reinterpret_cast<float*>(smem + G_STK);
            tmem_ld32(tmem + lane_off + 0 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) stq[(cb * 32 + j) * kD + l] = r[j];
            // dW and dv: lanes l and l ^ 1 trade one value per column pair, so
            // that each lane writes two adjacent entries of one column (the
            // even lane column j, the odd lane column j + 1): 4-byte stores,
            // two rows per warp instruction
            const bool odd = (lane & 1) != 0;
            const int l2 = l & ~1;
            tmem_ld32(tmem + lane_off + 64 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? r[j] : r[j + 1], 1);
                const float lo = odd ? recv : r[j], hi = odd ? r[j + 1] : recv;
                *reinterpret_cast<uint32_t*>(a.dW + rb + (size_t)(cb * 32 + j + (odd ? 1 : 0)) * kD +
                                             l2) = pack_bf16(-lo, -hi);
            }
            tmem_ld32(tmem + lane_off + 128 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) stk[(cb * 32 + j) * kD + l] = r[j];
            // D4: lanes 0-63 need columns 0-63 (dAqk), lanes 64-127 columns 64-127 (dTv)
            {
                const size_t cc = (size_t)crow * kC * kC;
                const int c4 = (q < 2 ? 0 : 2) + half;
                tmem_ld32(tmem + lane_off + 256 + c4 * 32, r);
                if (q < 2) {  // dAqk row i (bf16), masked to j <= i
                    const int i = l;
                    __nv_bfloat16* dst = a.dAqk + cc + (size_t)i * kC + c4 * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = (c4 * 32 + j) <= i ? r[j] : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        *reinterpret_cast<uint4*>(dst + j) =
                            make_uint4(pack_bf16(r[j], r[j + 1]), pack_bf16(r[j + 2], r[j + 3]),
                                       pack_bf16(r[j + 4], r[j + 5]), pack_bf16(r[j + 6], r[j + 7]));
                } else {  // dTv row i (fp32), masked to j < i
                    const int i = l - 64;
                    float* dst = a.dTv + cc + (size_t)i * kC + (c4 - 2) * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = ((c4 - 2) * 32 + j) < i ? r[j] : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + j) =
                            make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
                }
            }
            // D5: lane = v, columns m = 32*cb .. 32*cb+31
            tmem_ld32(tmem + lane_off + 192 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? r[j] : r[j + 1], 1);
                const float lo = odd ? recv : r[j], hi = odd ? r[j + 1] : recv;
                const int m = cb * 32 + j + (odd ? 1 : 0);
                const float bt = beta_s[m];
                if ((DW == kD || l2 < DW) && m < len)
                    *reinterpret_cast<uint32_t*>(a.dv + (((size_t)trow + m) * a.HV + hv) * DW + l2) =
                        pack_bf16(bt * lo, bt * hi);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int m = cb * 32 + j;
                const uint32_t voff =
                    G_DV + vbuf(it & 1) + (l >> 6) * 16384 + sw128_offset(m, l & 63);
                r[j] *= __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + voff));
            }
            // dbv[m] = sum over v of r: lane j ends with row cb*32 + j of this quadrant
            dbv_part[q * 64 + cb * 32 + lane] = warp_sum_scatter<32>(r);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0 && ok) {   // dQh and dKb from their staging tiles
            tma_store_2d(&tm_dqh, smem + G_STQ, 0, row);
            tma_store_2d(&tm_dkb, smem + G_STK, 0, row);
            bulk_commit_group();
        }
        // this v buffer has been read: the v tile two chunks ahead loads into it
        if (tid == 0 && ok && next + (int)gridDim.x < total) issue_v(next + gridDim.x);
        if (tid < kD)
            a.dgam[(size_t)crow * kD + tid] = dg_part[tid] + dg_part[kD + tid];
        if (tid < 64) {
            const int m = tid;
            a.dbv[(size_t)row + m] =
                (dbv_part[m] + dbv_part[64 + m]) + (dbv_part[128 + m] + dbv_part[192 + m]);
        }
        // partial sums, beta and TMEM are reused by the next chunk
        if (!__syncthreads_and(ok)) break;
    }
    // loads issued for chunks the loop did not reach (after an error) land
    // before shared memory is released
    if (tid == 0) {
        bulk_wait_all();   // the output stores complete
        for (; sd_waited < sd_issued; ++sd_waited) wait_bar_drain(bar_sd, sd_waited & 1);
        for (; main_waited < main_issued; ++main_waited) wait_bar_drain(bar_tma, main_waited & 1);
        for (; v_waited < v_issued; ++v_waited)
            wait_bar_drain((v_waited & 1) ? bar_v1 : bar_v, (v_waited >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// The contractions over V in two-term precision, for the backward with an
// upstream final-state gradient.  dS then carries that gradient (of the size
// of the inputs) back through the chunks, and products of dS, delta and Kb
// with single bf16 operands lose too much: the parts of dk and dbeta they
// feed cancel to values far smaller than their terms.  Here dS, delta and Kb
// come as bf16 high + low parts (x = hi + lo, about 16 mantissa bits) and
// each of their products takes three terms (hi hi + lo hi + hi lo):
//     ddelta^T = dS^T Kb^T + dO^T Aqk   (recomputed: the reverse pass's own
//                                        ddelta has single bf16 operands)
//     D3 = dS delta^T,  dgam = rowsum(dS o S0)
// and ddelta, split the same way, enters D2, D4 (bottom) and D5 as two
// terms.  S0, dO, v and T stay single bf16 operands.  One chunk at a time
// per CTA: every tile of a chunk loads at its start, with no overlap with
// the previous chunk, so that the shared-memory plan holds all of them.
// ===========================================================================
constexpr uint32_t P_S0 = 0;         // S0^T [128 v][128 k]: two 64-column boxes, 16 KB apart
constexpr uint32_t P_DS = 32768;     // dS^T high part, same layout
constexpr uint32_t P_DSL = 65536;    // dS^T low part; after the products, partial sums
constexpr uint32_t P_ODD = 98304;    // [dO; ddelta high], as in grad_v
constexpr uint32_t P_DV = 131072;    // Aqk [64 t][64 c] at +0, v at +8192 and +24576, T at +16384
constexpr uint32_t P_DT = 163840;    // delta^T high [128 v][64 c]
constexpr uint32_t P_DTL = 180224;   // delta^T low
constexpr uint32_t P_LO = 196608;    // Kb high at +0 / +16384, Kb low at +8192 / +24576 (one
                                     // 64-column box each); then ddelta low at +8192 / +24576
constexpr uint32_t P_BAR = 229376;
constexpr uint32_t PX_TX = 3 * 32768 + 16384 + 2 * 16384 + 32768 + 8192 + 16384 + 8192;
constexpr uint32_t PX_SMEM = P_BAR + 64 + 1024;
static_assert(PX_SMEM <= 232448, "the two-term contraction kernel exceeds the shared memory limit");
static_assert(P_DSL % 1024 == 0 && P_ODD % 1024 == 0 && P_DV % 1024 == 0 && P_DT % 1024 == 0 &&
                  P_DTL % 1024 == 0 && P_LO % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte aligned bases");

template <int DW, bool VL>
__global__ void __launch_bounds__(kGradThreads, 1)
grad_v_px_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_dh,
                 const __grid_constant__ CUtensorMap tm_dhl, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_dl,
                 const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_kbl,
                 const __grid_constant__ CUtensorMap tm_aqk, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_t, GradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(smem + P_BAR);   // every tile of the chunk
    uint64_t* bar_a = bar_ld + 1;                                     // ddelta, D1, D3
    uint64_t* bar_b = bar_ld + 2;                                     // D2, D4, D5
    uint64_t* bar_fin = bar_ld + 3;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_ld + 4);
    float* dbv_part = reinterpret_cast<float*>(smem + P_DSL);   // [4 lane quadrants][64]
    float* dg_part = dbv_part + 4 * 64;                          // [2 halves][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NT = a.NT, total = a.BH * NT;   // CTA i takes chunks i, i + grid, ...
    int issued = 0, waited = 0;               // thread 0's loads (each waited for before exit)
    auto issue = [&](int ch) {
        const int nn = ch % NT, bb = ch / NT, hvv = bb % a.HV;
        const int rw = bb * a.T + nn * kC, tr = tok_row((VL ? a.ctab : nullptr), bb / a.HV, a.T, nn);
        mbar_arrive_expect_tx(bar_ld, PX_TX);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            tma_load_2d(smem + P_S0 + hb * 16384, &tm_h, bar_ld, 64 * hb, ch * kD);
            tma_load_2d(smem + P_DS + hb * 16384, &tm_dh, bar_ld, 64 * hb, ch * kD);
            tma_load_2d(smem + P_DSL + hb * 16384, &tm_dhl, bar_ld, 64 * hb, ch * kD);
            tma_load_3d(smem + P_ODD + hb * 16384, &tm_do, bar_ld, 64 * hb, hvv, tr);
            tma_load_2d(smem + P_LO + hb * 16384, &tm_kb, bar_ld, 64 * hb, rw);
            tma_load_2d(smem + P_LO + 8192 + hb * 16384, &tm_kbl, bar_ld, 64 * hb, rw);
            tma_load_3d(smem + P_DV + 8192 + hb * 16384, &tm_v, bar_ld, 64 * hb, hvv, tr);
        }
        tma_load_2d(smem + P_DT, &tm_d, bar_ld, 0, ch * kD);
        tma_load_2d(smem + P_DTL, &tm_dl, bar_ld, 0, ch * kD);
        tma_load_2d(smem + P_DV, &tm_aqk, bar_ld, 0, ch * kC);
        tma_load_2d(smem + P_DV + 16384, &tm_t, bar_ld, 0, ch * kC);
        ++issued;
    };

    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_a, 1);
        mbar_init(bar_b, 1);
        mbar_init(bar_fin, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t id64 = idesc_bf16_f32(128, 64);
    const uint32_t s0 = smem_u32(smem + P_S0), ds = smem_u32(smem + P_DS),
                   dsl = smem_u32(smem + P_DSL), odd = smem_u32(smem + P_ODD),
                   dvb = smem_u32(smem + P_DV), dt = smem_u32(smem + P_DT),
                   dtl = smem_u32(smem + P_DTL), lo = smem_u32(smem + P_LO);
    // all 8 warps, two per TMEM lane quadrant, splitting the columns
    const int q = warp & 3, half = warp >> 2;
    const int l = q * 32 + lane;   // TMEM lane: v for ddelta^T and D5, k for D1-D3, row for D4
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    bool ok = true;

#pragma unroll 1
    for (int it = 0, chunk = blockIdx.x; chunk < total; ++it, chunk += gridDim.x) {
        const uint32_t ph = it & 1;
        const int n = chunk % NT, bh = chunk / NT;
        const int b = bh / a.HV, hv = bh % a.HV;
        const int row = bh * a.T + n * kC;
        const int trow = tok_row((VL ? a.ctab : nullptr), b, a.T, n);
        const int len = tok_len((VL ? a.ctab : nullptr), n);   // rows past it belong to the next sequence
        if (tid == 0) {
            issue(chunk);
            if (wait_bar(bar_ld, ph, 51)) {
                ++waited;
                tc_fence_after();
                // ddelta^T [v][c] -> TMEM columns 384..447: dS^T read K-major
                // (rows v), Kb K-major (rows c), three terms
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + 384, sdesc_sw128(ds + ko), sdesc_sw128(lo + ko), id64, kk > 0);
                    mma_bf16(tmem + 384, sdesc_sw128(dsl + ko), sdesc_sw128(lo + ko), id64, 1);
                    mma_bf16(tmem + 384, sdesc_sw128(ds + ko), sdesc_sw128(lo + 8192 + ko), id64, 1);
                }
                // + dO^T Aqk: dO read MN-major (v blocks 16 KB apart), Aqk MN-major
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + 384, sdesc_mn_sw128(odd + kk * 2048, 16384),
                             sdesc_mn_sw128(dvb + kk * 2048, 8192), id64 | kAMajorMN | kBMajorMN, 1);
                // D1 = S0 dO^T -> columns 0..63; D3 = dS delta^T -> 128..191 (three terms).
                // S0 and dS are stored transposed (rows v): A operands read
                // MN-major, K = v advancing 16 rows per step
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t ads = sdesc_mn_sw128(ds + kk * 2048, 16384);
                    const uint64_t bdt = sdesc_mn_sw128(dt + kk * 2048, 16384);
                    mma_bf16(tmem + 0, sdesc_mn_sw128(s0 + kk * 2048, 16384), sdesc_sw128(odd + ko),
                             id64 | kAMajorMN, kk > 0);
                    mma_bf16(tmem + 128, ads, bdt, id64 | kAMajorMN | kBMajorMN, kk > 0);
                    mma_bf16(tmem + 128, sdesc_mn_sw128(dsl + kk * 2048, 16384), bdt,
                             id64 | kAMajorMN | kBMajorMN, 1);
                    mma_bf16(tmem + 128, ads, sdesc_mn_sw128(dtl + kk * 2048, 16384),
                             id64 | kAMajorMN | kBMajorMN, 1);
                }
                mma_commit(bar_a);
            } else {
                ok = false;
            }
        }
        __syncwarp();
        float r[32];
        ok = ok && wait_bar_warp(bar_a, ph, 52);
        tc_fence_after();
        if (ok) {
            // ddelta (row c, column v = l) as high and low bf16 parts: the high
            // part into rows 64..127 of the [dO; ddelta] tile, the low part
            // over Kb's (read by the products above) in the same layout
            tmem_ld32(tmem + lane_off + 384 + 32 * half, r);
            const uint32_t box = (uint32_t)(l >> 6) * 16384;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint32_t off = 8192 + box + sw128_offset(32 * half + j, l & 63);
                const __nv_bfloat16 hi = __float2bfloat16_rn(r[j]);
                *reinterpret_cast<__nv_bfloat16*>(smem + P_ODD + off) = hi;
                *reinterpret_cast<__nv_bfloat16*>(smem + P_LO + off) =
                    __float2bfloat16_rn(r[j] - __bfloat162float(hi));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0 && ok) {
            const uint32_t tt = dvb + 16384;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint64_t as0 = sdesc_mn_sw128(s0 + kk * 2048, 16384);
                const uint64_t bv = sdesc_sw128(dvb + 8192 + ko);
                // D2 = S0 ddelta^T -> columns 64..127 (two terms)
                mma_bf16(tmem + 64, as0, sdesc_sw128(odd + 8192 + ko), id64 | kAMajorMN, kk > 0);
                mma_bf16(tmem + 64, as0, sdesc_sw128(lo + 8192 + ko), id64 | kAMajorMN, 1);
                // D4 = [dO; ddelta] [delta; v]^T: delta^T -> 256..319 (lanes 0..63
                // used), v -> 320..383 (lanes 64..127 used), the low part of
                // ddelta as a second term whose rows 0..63 (Kb's high part)
                // land in the unused lanes
                mma_bf16(tmem + 256, sdesc_sw128(odd + ko), sdesc_mn_sw128(dt + kk * 2048, 16384),
                         id64 | kBMajorMN, kk > 0);
                mma_bf16(tmem + 320, sdesc_sw128(odd + ko), bv, id64, kk > 0);
                mma_bf16(tmem + 320, sdesc_sw128(lo + ko), bv, id64, 1);
            }
            // D5 = ddelta^T T -> 192..255 (two terms): ddelta read MN-major, T MN-major
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bt = sdesc_mn_sw128(tt + kk * 2048, 8192);
                mma_bf16(tmem + 192, sdesc_mn_sw128(odd + 8192 + kk * 2048, 16384), bt,
                         id64 | kAMajorMN | kBMajorMN, kk > 0);
                mma_bf16(tmem + 192, sdesc_mn_sw128(lo + 8192 + kk * 2048, 16384), bt,
                         id64 | kAMajorMN | kBMajorMN, 1);
            }
            mma_commit(bar_b);
        }
        __syncwarp();
        ok = ok && wait_bar_warp(bar_b, ph, 53);
        tc_fence_after();
        // dgam[k] = sum_v (dS_hi + dS_lo)[v][k] S0[v][k]; thread (k = l, half)
        // sums rows v in [64 half, 64 half + 64)
        float dgp = 0.f;
        if (ok) {
            const uint32_t kb = (uint32_t)(l >> 6) * 16384;
#pragma unroll 8
            for (int vv = 0; vv < 64; ++vv) {
                const uint32_t off = kb + sw128_offset(64 * half + vv, l & 63);
                const float dsv =
                    __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + P_DS + off)) +
                    __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + P_DSL + off));
                dgp += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + P_S0 + off)) *
                       dsv;
            }
        }
        __syncthreads();   // the dS low tile is read: the partial sums go there
        dg_part[half * kD + l] = dgp;
        if (ok) {
            const size_t rb = (size_t)row * kD;
            const int cb = half;  // columns 32*cb .. 32*cb+31 of D1-D3 and D5
            tmem_ld32(tmem + lane_off + 0 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) a.dQh[rb + (size_t)(cb * 32 + j) * kD + l] = r[j];
            tmem_ld32(tmem + lane_off + 64 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                a.dW[rb + (size_t)(cb * 32 + j) * kD + l] = __float2bfloat16_rn(-r[j]);
            tmem_ld32(tmem + lane_off + 128 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) a.dKb[rb + (size_t)(cb * 32 + j) * kD + l] = r[j];
            {
                const size_t cc = (size_t)chunk * kC * kC;
                const int c4 = (q < 2 ? 0 : 2) + half;
                tmem_ld32(tmem + lane_off + 256 + c4 * 32, r);
                if (q < 2) {  // dAqk row i (bf16), masked to j <= i
                    const int i = l;
                    __nv_bfloat16* dst = a.dAqk + cc + (size_t)i * kC + c4 * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = (c4 * 32 + j) <= i ? r[j] : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        *reinterpret_cast<uint4*>(dst + j) =
                            make_uint4(pack_bf16(r[j], r[j + 1]), pack_bf16(r[j + 2], r[j + 3]),
                                       pack_bf16(r[j + 4], r[j + 5]), pack_bf16(r[j + 6], r[j + 7]));
                } else {  // dTv row i (fp32), masked to j < i
                    const int i = l - 64;
                    float* dst = a.dTv + cc + (size_t)i * kC + (c4 - 2) * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = ((c4 - 2) * 32 + j) < i ? r[j] : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + j) =
                            make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
                }
            }
            // D5: lane = v, columns m = 32*cb .. 32*cb+31
            tmem_ld32(tmem + lane_off + 192 + cb * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int m = cb * 32 + j;
                const float bt =
                    m < len ? __bfloat162float(a.beta[((size_t)trow + m) * a.HV + hv]) : 0.f;
                if ((DW == kD || l < DW) && m < len)
                    a.dv[(((size_t)trow + m) * a.HV + hv) * DW + l] = __float2bfloat16_rn(bt * r[j]);
                const uint32_t voff = P_DV + 8192 + (l >> 6) * 16384 + sw128_offset(m, l & 63);
                r[j] *= __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + voff));
            }
            // dbv[m] = sum over v of r: lane j ends with row cb*32 + j of this quadrant
            dbv_part[q * 64 + cb * 32 + lane] = warp_sum_scatter<32>(r);
        }
        __syncthreads();
        if (ok && tid < kD) a.dgam[(size_t)chunk * kD + tid] = dg_part[tid] + dg_part[kD + tid];
        if (ok && tid < 64)
            a.dbv[(size_t)row + tid] =
                (dbv_part[tid] + dbv_part[64 + tid]) + (dbv_part[128 + tid] + dbv_part[192 + tid]);
        // the next chunk's loads overwrite every tile and the partial sums
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;
        tc_fence_after();
    }
    // a load issued for a chunk the loop did not finish (after an error)
    // lands before shared memory is released; every product completes before
    // TMEM is
    if (tid == 0) {
        for (; waited < issued; ++waited) wait_bar_drain(bar_ld, waited & 1);
        mma_commit(bar_fin);
        wait_bar_drain(bar_fin, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// Intra-chunk quantities on tensor cores (K3 row L2 steps (1)-(3) plus the
// operands of the state passes), one chunk of one head at a time per CTA of
// 256 threads.  Shared memory stays under half an SM's, so two CTAs share an
// SM and one's dependent phases (barriers, MMA and TMA waits, the triangular
// inverse) overlap the other's work.
//   (1) G_rel = cumsum of max(g, -5) inside each 16-row block, as one MMA:
//       a constant 0/1 matrix (row r has ones at 16 floor(r/16) < r' <= r)
//       times the clamped g tile.  The product has M = 128: rows 64-127
//       repeat rows 0-63, so every TMEM lane quadrant holds a copy of the
//       chunk's rows.  Block offsets G_b (G at each block's first row) and
//       G_last follow from the block ends and block-start gates.
//   (2) A, Aqk: the pairwise decay exp(G_i - G_j) is factored per 16-row
//       block R with reference row b = 16R:  exp(G_i - G_b) <= 1 on the left,
//       exp(G_b - G_j) on the right (<= 1 for earlier blocks, <= e^75 inside
//       the block since g >= -5), so no factor overflows fp32/bf16.
//       D_R = Left Right_R^T (M=128, N=16(R+1)), where Left row 32R + 16s + u
//       holds token 16R+u (s=0: k, s=1: q) times exp(G - G_b), so TMEM warp
//       quadrant R holds exactly block R's rows.  The product runs in two
//       64-channel halves through one Left/Right buffer.
//   (3) T = (I + A)^{-1} (fp32, blocked forward substitution),
//       W = (T diag beta) Khat and U = (T diag beta) V as row-major products
//       (M = 128: the T diag beta operand is stored twice), Khat and V read
//       MN-major from their tiles.
// Elementwise work runs with one thread per (row, 32 key channels); Qh and
// Kb are written in place over the q and k tiles.  Every output leaves
// through a TMA store of its shared-memory tile (W, Qh, U, Kb, Aqk) or as
// 16-byte rows (T as bf16 high and low parts, when asked for) and gam.
// ===========================================================================
constexpr uint32_t J_L = 0;          // [128][64] bf16 block-lower-triangular ones (constant)
constexpr uint32_t J_K = 16384;      // k tile -> Kb (in place) -> Aqk staging
constexpr uint32_t J_Q = 32768;      // q tile -> Qh (in place) -> v tile -> U staging
constexpr uint32_t J_G = 49152;      // g tile (clamped in place) -> Khat -> W staging
constexpr uint32_t J_LR = 65536;     // Left half [128][64] + Right half [160][64]; then A, T
constexpr uint32_t J_RIGHT = J_LR + 16384;
constexpr int kAS = 68;              // row stride (floats) of A and T: rows stay 16-byte aligned
constexpr uint32_t J_A = J_LR;                       // fp32 [64][kAS]
constexpr uint32_t J_T = J_LR + 64 * kAS * 4;        // fp32 [64][kAS]
constexpr uint32_t J_TB = J_LR;      // T diag(beta), bf16 [128][64] (rows 64-127 repeat), over A
constexpr uint32_t J_SCR = J_LR;     // block ends and block-start gates, fp32 [2][4][128]
constexpr uint32_t J_BETA = J_LR + 36864;            // fp32 [64]
constexpr uint32_t J_C = J_BETA + 256;               // exp(G_b) [4][128], exp(G_last-G_b) [4][128], F [6][128]
constexpr uint32_t J_BAR = J_C + 14 * 512;
constexpr uint32_t INTRA_SMEM = J_BAR + 64 + 1024;
static_assert(J_T + 64 * kAS * 4 <= J_BETA, "A and T overflow the Left/Right area");
static_assert(INTRA_SMEM <= 115712, "two intra CTAs must fit one SM's shared memory");
static_assert(J_L % 1024 == 0 && J_K % 1024 == 0 && J_Q % 1024 == 0 && J_G % 1024 == 0 &&
                  J_LR % 1024 == 0 && J_RIGHT % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte aligned bases");

// slot of F(R, Rr) = exp(G_b(Rr) - G_b(R)) for Rr > R among the six pairs
__host__ __device__ constexpr int f_slot(int R, int Rr) { return R * (7 - R) / 2 + (Rr - R - 1); }

constexpr int kIntraThreads = 256;

// first row of Right_R in the stacked operand, which is also the first TMEM
// column of D_R: sum_{J<R} 16 (J+1)
__host__ __device__ constexpr uint32_t right_col(int R) { return 8u * (uint32_t)(R * (R + 1)); }

struct IntraArgs {
    int T, H, HV, NT, BH;
    int D;                     // K = V of the tensors (64 or 128); the kernel works at 128
    float scale;
    int qkn;                   // L2-normalise the q and k tiles first
    const __nv_bfloat16* beta;
    __nv_bfloat16 *T2, *Tlo;   // null: T is not kept (plain forward)
    // low parts (x - bf16(x)) of U and Kb, [BH*T][128] like their arrays, or
    // null (only the backward with an upstream final-state gradient asks)
    __nv_bfloat16 *Ulo, *Kblo;
    float* gam;
    const int* ctab;           // packed sequences: the chunk table, or null
};

template <int R>
__device__ __forceinline__ void intra_read_block(uint32_t taddr, float* out /* 64 */) {
    // lanes of warp quadrant R: columns of D_R (16(R+1) of them)
    float r[32];
    constexpr int N = 16 * (R + 1);
#pragma unroll
    for (int cb = 0; cb < (N + 31) / 32; ++cb) {
        tmem_ld32(taddr + cb * 32, r);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (cb * 32 + j < N) out[cb * 32 + j] = r[j];
    }
#pragma unroll
    for (int j = N; j < 64; ++j) out[j] = 0.f;
}

// LO: also write the low parts of U and Kb (a.Ulo, a.Kblo); a separate
// instantiation, so that the plain one keeps its registers.
template <bool LO, bool VL>
__global__ void __launch_bounds__(kIntraThreads, 2)
intra_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_q2,
                const __grid_constant__ CUtensorMap tm_u2, const __grid_constant__ CUtensorMap tm_kb2,
                const __grid_constant__ CUtensorMap tm_aqk2, IntraArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar_kqg = reinterpret_cast<uint64_t*>(smem + J_BAR);   // k, q, g tiles
    uint64_t* bar_v = bar_kqg + 1;                                     // v tile
    uint64_t* bar_g = bar_kqg + 2;                                     // G_rel product
    uint64_t* bar_a0 = bar_kqg + 3;                                    // D, channels 0-63
    uint64_t* bar_a1 = bar_kqg + 4;                                    // D, channels 64-127
    uint64_t* bar_w = bar_kqg + 5;                                     // W and U products
    uint64_t* bar_fin = bar_kqg + 6;                                   // every product issued
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_kqg + 7);
    float* sA = reinterpret_cast<float*>(smem + J_A);
    float* sT = reinterpret_cast<float*>(smem + J_T);
    float* sBeta = reinterpret_cast<float*>(smem + J_BETA);
    float* sGend = reinterpret_cast<float*>(smem + J_SCR);   // [4][128] G_rel at block ends
    float* sG0 = sGend + 4 * kD;                              // [4][128] clamped g at block starts
    float* sEGb = reinterpret_cast<float*>(smem + J_C);      // [4][128] exp(G_b)
    float* sELb = sEGb + 4 * kD;                              // [4][128] exp(G_last - G_b)
    float* sF = sELb + 4 * kD;                                // [6][128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.BH * a.NT;   // chunks; CTA i takes chunks i, i + grid, ...
    // elementwise role: chunk row r (TMEM lane quadrant qd holds rows
    // 32 (qd & 1) .. + 31) and channel quarter jq: channels 16 jq .. + 15 and
    // 64 + 16 jq .. + 15
    const int qd = warp & 3;
    const int r = 32 * (qd & 1) + lane, R = r >> 4, u = r & 15;
    const int jq = (qd >> 1) + 2 * (warp >> 2);
    const uint32_t tlane = (uint32_t)(32 * qd) << 16;

    // token row of chunk ch, its value head and key head
    auto coords = [&](int ch, int& trow, int& hv, int& h) {
        const int nn = ch % a.NT, bb = ch / a.NT;
        hv = bb % a.HV;
        h = hv / (a.HV / a.H);
        trow = tok_row((VL ? a.ctab : nullptr), bb / a.HV, a.T, nn);
    };
    // thread 0's counts of issued and consumed loads (every load is waited for
    // before the CTA exits)
    int kqg_issued = 0, v_issued = 0, kqg_waited = 0, v_waited = 0;
    auto issue_kqg = [&](int ch) {
        int trow, hv, h;
        coords(ch, trow, hv, h);
        mbar_arrive_expect_tx(bar_kqg, 3 * 16384);
        tma_load_3d(smem + J_K, &tm_k, bar_kqg, 0, h, trow);
        tma_load_3d(smem + J_K + 8192, &tm_k, bar_kqg, 64, h, trow);
        tma_load_3d(smem + J_Q, &tm_q, bar_kqg, 0, h, trow);
        tma_load_3d(smem + J_Q + 8192, &tm_q, bar_kqg, 64, h, trow);
        tma_load_3d(smem + J_G, &tm_g, bar_kqg, 0, hv, trow);
        tma_load_3d(smem + J_G + 8192, &tm_g, bar_kqg, 64, hv, trow);
        ++kqg_issued;
    };
    auto issue_v = [&](int ch) {
        int trow, hv, h;
        coords(ch, trow, hv, h);
        mbar_arrive_expect_tx(bar_v, 16384);
        tma_load_3d(smem + J_Q, &tm_v, bar_v, 0, hv, trow);
        tma_load_3d(smem + J_Q + 8192, &tm_v, bar_v, 64, hv, trow);
        ++v_issued;
    };
    // the chunk's tiles into L2 ahead of their loads
    auto prefetch = [&](int ch) {
        int trow, hv, h;
        coords(ch, trow, hv, h);
        tma_prefetch_3d(&tm_k, 0, h, trow);
        tma_prefetch_3d(&tm_q, 0, h, trow);
        tma_prefetch_3d(&tm_g, 0, hv, trow);
        tma_prefetch_3d(&tm_v, 0, hv, trow);
        if (a.D > 64) {   // at D = 64 the upper boxes lie past the rows
            tma_prefetch_3d(&tm_k, 64, h, trow);
            tma_prefetch_3d(&tm_q, 64, h, trow);
            tma_prefetch_3d(&tm_g, 64, hv, trow);
            tma_prefetch_3d(&tm_v, 64, hv, trow);
        }
    };
    auto load_beta = [&](int ch) {   // 0 past a packed sequence's end
        int trow, hv, h;
        coords(ch, trow, hv, h);
        return tid < tok_len((VL ? a.ctab : nullptr), ch % a.NT)
                   ? __bfloat162float(a.beta[((size_t)trow + tid) * a.HV + hv])
                   : 0.f;
    };

    if (tid == 0) {
        for (int i = 0; i < 7; ++i) mbar_init(bar_kqg + i, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, 256);
        tmem_relinquish();
    }
    // the constant block-lower-triangular operand: row i (token r = i & 63)
    // has ones at 16 floor(r / 16) < r' <= r; thread t fills four 8-column units
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
        const int unit = tid + 256 * k4, i = unit >> 3, o = unit & 7, rr = i & 63;
        const int lo = (rr & ~15) + 1;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = 8 * o + e;
            x[e] = (c >= lo && c <= rr) ? 1.f : 0.f;
        }
        *reinterpret_cast<uint4*>(smem + J_L + sw128_offset(i, 8 * o)) = pack8(x);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (tid == 0 && (int)blockIdx.x < total) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_v);
        issue_kqg(blockIdx.x);
    }
    float beta_next = (tid < kC && (int)blockIdx.x < total) ? load_beta(blockIdx.x) : 0.f;
    bool ok = true;

#pragma unroll 1
    for (int it = 0, chunk = blockIdx.x; chunk < total; ++it, chunk += gridDim.x) {
    const uint32_t ph = it & 1;
    const int next = chunk + gridDim.x;
    const int n = chunk % a.NT, bh = chunk / a.NT;
    const int row0 = bh * a.T + n * kC;       // row in the [BH*T] workspace arrays
    const int crow = chunk;                   // chunk index
    const int len = tok_len((VL ? a.ctab : nullptr), n);       // valid rows (a partial chunk of a packed batch)
    if (tid == 0 && next < total) prefetch(next);
    if (tid < kC) {
        sBeta[tid] = tid < len ? beta_next : 0.f;                 // read after later barriers
        if (next < total) beta_next = load_beta(next);            // in flight meanwhile
    }
    {
        const bool got = wait_bar_warp(bar_kqg, ph, 31);
        if (got && tid == 0) ++kqg_waited;
        ok = ok && got;
    }
    if (len < kC) {
        // rows past the end of a packed sequence: q = k = 0, g = 0 (with
        // beta = 0 they leave every output of the valid rows unchanged)
        zero_tile_rows(smem + J_K, len, tid, kIntraThreads);
        zero_tile_rows(smem + J_Q, len, tid, kIntraThreads);
        zero_tile_rows(smem + J_G, len, tid, kIntraThreads);
        __syncthreads();
    }

    // ---- (1) clamp the g tile in place (1024 units of 8 bf16); with qkn,
    // normalise the rows of the k and q tiles in place ----
    if (a.qkn) {
        l2norm_tile_rows(smem + J_K, tid, kIntraThreads);
        l2norm_tile_rows(smem + J_Q, tid, kIntraThreads);
    }
    {
        const __nv_bfloat162 floor2 = __floats2bfloat162_rn(kGateFloor, kGateFloor);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            uint4* p = reinterpret_cast<uint4*>(smem + J_G) + tid + 256 * k4;
            uint4 v4 = *p;
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&v4);
#pragma unroll
            for (int e = 0; e < 4; ++e) h2[e] = __hmax2(h2[e], floor2);
            *p = v4;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // G_rel = Lrel . gclamp: M = 128 (rows 64-127 repeat), N = 128 channels, K = 64 rows
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, 128) | kBMajorMN;
        const uint32_t l = smem_u32(smem + J_L), gt = smem_u32(smem + J_G);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, sdesc_sw128(l + kk * 32), sdesc_mn_sw128(gt + kk * 2048, 8192), id,
                     kk > 0);
        mma_commit(bar_g);
    }
    ok = ok && wait_bar_warp(bar_g, ph, 35);
    tc_fence_after();
    // this thread's 32 block-relative cumsums
    float Gr[32];
    {
        float x[16];
        tmem_ld16(tmem + tlane + 16 * jq, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) Gr[e] = x[e];
        tmem_ld16(tmem + tlane + 64 + 16 * jq, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) Gr[16 + e] = x[e];
    }
    // block ends and block-start gates for the per-block constants
    if (u == 15) {
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            *reinterpret_cast<float4*>(sGend + R * kD + 16 * jq + e) =
                make_float4(Gr[e], Gr[e + 1], Gr[e + 2], Gr[e + 3]);
            *reinterpret_cast<float4*>(sGend + R * kD + 64 + 16 * jq + e) =
                make_float4(Gr[16 + e], Gr[17 + e], Gr[18 + e], Gr[19 + e]);
        }
    } else if (u == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float x[8];
                unpack8(*reinterpret_cast<const uint4*>(smem + J_G + hh * 8192 +
                                                        sw128_offset(r, 16 * jq + 8 * e)),
                        x);
                float* dst = sG0 + R * kD + 64 * hh + 16 * jq + 8 * e;
                *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // per (block, channel) constants: thread (c, part) with c = tid % 128
    {
        const int c = tid & (kD - 1);
        float gb[4];
        gb[0] = sG0[c];
#pragma unroll
        for (int p = 1; p < 4; ++p) gb[p] = gb[p - 1] + sGend[(p - 1) * kD + c] + sG0[p * kD + c];
        const float glast = gb[3] + sGend[3 * kD + c];
        if (tid < kD) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                sEGb[p * kD + c] = __expf(gb[p]);
                sELb[p * kD + c] = __expf(glast - gb[p]);
            }
            a.gam[(size_t)crow * kD + c] = __expf(glast);
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int pr = p + 1; pr < 4; ++pr) sF[f_slot(p, pr) * kD + c] = __expf(gb[pr] - gb[p]);
        }
    }
    __syncthreads();

    // ---- operands, in two 64-channel halves through one Left/Right buffer:
    // Left (k E, q E), Right_Rr (Rr >= R), Khat into the g area, Qh and Kb in
    // place over the q and k tiles ----
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        if (hh == 1) {
            // the first half's product has read the Left/Right buffer
            ok = ok && wait_bar_warp(bar_a0, ph, 36);
            tc_fence_after();
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int o = 2 * jq + e;                 // 8-channel unit within the half
            const int c0 = 64 * hh + 8 * o;           // first channel
            const uint32_t tile_off = hh * 8192 + sw128_offset(r, 8 * o);
            float kv[8], qv[8], egb[8], elb[8], E[8], Ei[8], x[8];
            unpack8(*reinterpret_cast<const uint4*>(smem + J_K + tile_off), kv);
            unpack8(*reinterpret_cast<const uint4*>(smem + J_Q + tile_off), qv);
            ld8f(sEGb + R * kD + c0, egb);
            ld8f(sELb + R * kD + c0, elb);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float gr = Gr[16 * hh + 8 * e + i];
                E[i] = __expf(gr);       // exp(G - G_b) <= 1
                Ei[i] = __expf(-gr);     // exp(G_b - G) in [1, e^75]
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = kv[i] * E[i];
            *reinterpret_cast<uint4*>(smem + J_LR + sw128_offset(32 * R + u, 8 * o)) = pack8(x);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = qv[i] * E[i];
            *reinterpret_cast<uint4*>(smem + J_LR + sw128_offset(32 * R + 16 + u, 8 * o)) = pack8(x);
#pragma unroll
            for (int i = 0; i < 8; ++i) Ei[i] *= kv[i];                       // k exp(G_b - G)
            *reinterpret_cast<uint4*>(smem + J_RIGHT + sw128_offset(right_col(R) + r, 8 * o)) =
                pack8(Ei);
#pragma unroll
            for (int Rr = 1; Rr < 4; ++Rr) {
                if (Rr <= R) continue;
                float f8[8];
                ld8f(sF + f_slot(R, Rr) * kD + c0, f8);
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = Ei[i] * f8[i];
                *reinterpret_cast<uint4*>(smem + J_RIGHT + sw128_offset(right_col(Rr) + r, 8 * o)) =
                    pack8(x);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = kv[i] * E[i] * egb[i];          // Khat = k exp(G)
            *reinterpret_cast<uint4*>(smem + J_G + tile_off) = pack8(x);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = qv[i] * E[i] * egb[i] * a.scale;  // Qh
            *reinterpret_cast<uint4*>(smem + J_Q + tile_off) = pack8(x);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = Ei[i] * elb[i];                 // Kb = k exp(G_last - G)
            *reinterpret_cast<uint4*>(smem + J_K + tile_off) = pack8(x);
            if (LO)
                *reinterpret_cast<uint4*>(a.Kblo + (size_t)(row0 + r) * kD + c0) = pack8_lo(x);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0 && ok) {
            // D (+)= Left_h Right_h^T over this half's 64 channels, N = 160
            const uint32_t left = smem_u32(smem + J_LR), right = smem_u32(smem + J_RIGHT);
            const uint32_t id = idesc_bf16_f32(128, 160);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem, sdesc_sw128(left + kk * 32), sdesc_sw128(right + kk * 32), id,
                         (hh > 0 || kk > 0) ? 1u : 0u);
            mma_commit(hh == 0 ? bar_a0 : bar_a1);
            if (hh == 1) {
                // Qh and Kb are complete: out by TMA
                tma_store_2d(&tm_q2, smem + J_Q, 0, row0);
                tma_store_2d(&tm_q2, smem + J_Q + 8192, 64, row0);
                tma_store_2d(&tm_kb2, smem + J_K, 0, row0);
                tma_store_2d(&tm_kb2, smem + J_K + 8192, 64, row0);
                bulk_commit_group();
            }
        }
    }
    ok = ok && wait_bar_warp(bar_a1, ph, 32);
    tc_fence_after();
    if (tid == 0) {
        // the Qh and Kb stores have read their tiles: the v tile loads into
        // the q area, and the k area takes the Aqk staging tile
        bulk_wait_read_all();
        if (ok) issue_v(chunk);
    }
    __syncthreads();
    if (ok) {
        // warps R and R + 4 read block R (TMEM quadrant R); lanes 0-15 of warp R
        // write its A rows, lanes 16-31 of warp R + 4 its Aqk rows
        const int Rq = warp & 3;
        float d[64];
        const uint32_t taddr = tmem + ((uint32_t)(Rq * 32) << 16) + right_col(Rq);
        if (Rq == 0) intra_read_block<0>(taddr, d);
        else if (Rq == 1) intra_read_block<1>(taddr, d);
        else if (Rq == 2) intra_read_block<2>(taddr, d);
        else intra_read_block<3>(taddr, d);
        const int uu = lane & 15, i = 16 * Rq + uu;
        if (warp < 4 && lane < 16) {
            const float bi = sBeta[i];
#pragma unroll
            for (int j = 0; j < kC; j += 4)
                *reinterpret_cast<float4*>(sA + i * kAS + j) =
                    make_float4(j < i ? bi * d[j] : 0.f, j + 1 < i ? bi * d[j + 1] : 0.f,
                                j + 2 < i ? bi * d[j + 2] : 0.f, j + 3 < i ? bi * d[j + 3] : 0.f);
        } else if (warp >= 4 && lane >= 16) {
#pragma unroll
            for (int j = 0; j < kC; j += 8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (j + e <= i) ? a.scale * d[j + e] : 0.f;
                *reinterpret_cast<uint4*>(smem + J_K + sw128_offset(i, j)) = pack8(x);
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        tma_store_2d(&tm_aqk2, smem + J_K, 0, crow * kC);
        bulk_commit_group();
    }

    // ---- (3) T = (I + A)^{-1}, A strictly lower, in three levels: the four
    // 16 x 16 diagonal blocks by forward substitution (thread (B, jj) keeps
    // column jj of block B in registers); each 32 x 32 diagonal block as
    // [[T_a, 0], [-T_b (A_ba T_a), T_b]]; then T_10 = -T_11 (A_10 T_00).  A's
    // entries on and above the diagonal are stored zeros, so the dot products
    // run over whole float4s. ----
    if (tid < 64) {
        const int o = 16 * (tid >> 4), jj = tid & 15;
        float t[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) t[m] = m == jj ? 1.f : 0.f;
#pragma unroll
        for (int ii = 1; ii < 16; ++ii) {
            const float* arow = sA + (o + ii) * kAS + o;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < ii; m += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(arow + m);
                acc[0] += a4.x * t[m];
                acc[1] += a4.y * t[m + 1];
                acc[2] += a4.z * t[m + 2];
                acc[3] += a4.w * t[m + 3];
            }
            if (ii > jj) t[ii] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) sT[(o + m) * kAS + o + jj] = t[m];
    }
    __syncthreads();
    // 32-level, thread (i, j) for both diagonal 32-blocks RB: Y = A_ba T_a into
    // A's unused block above the diagonal (rows o + i, columns o + 16 + j);
    // T's blocks above the diagonal (that one, and T_01) are zero
    {
        const int i = tid >> 4, j = tid & 15;
#pragma unroll
        for (int RB = 0; RB < 2; ++RB) {
            const int o = 32 * RB;
            const float* arow = sA + (o + 16 + i) * kAS + o;
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(arow + m);
                y0 = fmaf(a4.x, sT[(o + m) * kAS + o + j], y0);
                y1 = fmaf(a4.y, sT[(o + m + 1) * kAS + o + j], y1);
                y0 = fmaf(a4.z, sT[(o + m + 2) * kAS + o + j], y0);
                y1 = fmaf(a4.w, sT[(o + m + 3) * kAS + o + j], y1);
            }
            sA[(o + i) * kAS + o + 16 + j] = y0 + y1;
            sT[(o + i) * kAS + o + 16 + j] = 0.f;
        }
#pragma unroll
        for (int rr = 0; rr < 32; rr += 8)   // T_01, rows 0..31, columns 32..63
            sT[(rr + (tid >> 5)) * kAS + 32 + (tid & 31)] = 0.f;
    }
    __syncthreads();
    // T_ba = -T_b Y
    {
        const int i = tid >> 4, j = tid & 15;
#pragma unroll
        for (int RB = 0; RB < 2; ++RB) {
            const int o = 32 * RB;
            const float* trow = sT + (o + 16 + i) * kAS + o + 16;
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(trow + m);
                y0 = fmaf(t4.x, sA[(o + m) * kAS + o + 16 + j], y0);
                y1 = fmaf(t4.y, sA[(o + m + 1) * kAS + o + 16 + j], y1);
                y0 = fmaf(t4.z, sA[(o + m + 2) * kAS + o + 16 + j], y0);
                y1 = fmaf(t4.w, sA[(o + m + 3) * kAS + o + 16 + j], y1);
            }
            sT[(o + 16 + i) * kAS + o + j] = -(y0 + y1);
        }
    }
    __syncthreads();
    // The two 32 x 32 x 32 products below: thread (rp, cp) owns rows 2rp,
    // 2rp + 1 and columns 2cp, 2cp + 1 of C = sign A B (row stride kAS
    // everywhere).  Per four k: two float4 loads of A rows (shared by a
    // half-warp) and four float2 loads of B (shared by the two half-warps)
    // feed 16 FMAs.
    auto mm32 = [&](const float* A, const float* B, float* C, float sign) {
        const int rp = 2 * warp + (lane >> 4), cp = lane & 15;
        const int i0 = 2 * rp, j0 = 2 * cp;
        const float* a0 = A + i0 * kAS;
        const float* a1 = a0 + kAS;
        float c00 = 0.f, c01 = 0.f, c10 = 0.f, c11 = 0.f;
#pragma unroll
        for (int m = 0; m < 32; m += 4) {
            const float4 p = *reinterpret_cast<const float4*>(a0 + m);
            const float4 q = *reinterpret_cast<const float4*>(a1 + m);
            const float pa[4] = {p.x, p.y, p.z, p.w}, qa[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 bv = *reinterpret_cast<const float2*>(B + (m + e) * kAS + j0);
                c00 = fmaf(pa[e], bv.x, c00);
                c01 = fmaf(pa[e], bv.y, c01);
                c10 = fmaf(qa[e], bv.x, c10);
                c11 = fmaf(qa[e], bv.y, c11);
            }
        }
        *reinterpret_cast<float2*>(C + i0 * kAS + j0) = make_float2(sign * c00, sign * c01);
        *reinterpret_cast<float2*>(C + (i0 + 1) * kAS + j0) = make_float2(sign * c10, sign * c11);
    };
    // X = A_10 T_00 into A's unused upper block (rows 0..31, columns 32..63)
    mm32(sA + 32 * kAS, sT, sA + 32, 1.f);
    __syncthreads();
    // T_10 = -T_11 X
    mm32(sT + 32 * kAS + 32, sA + 32, sT + 32 * kAS, -1.f);
    __syncthreads();
    // T (bf16 high and low parts) to global when kept; T*beta, twice, to the
    // A operand of the W and U products (over A, whose last reader was the
    // product above).  Thread t takes columns 8 (t % 8) .. + 7 of rows t / 8
    // and t / 8 + 32.
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int i = (tid >> 3) + 32 * half, ch = tid & 7, j0 = ch * 8;
        float t8[8], b8[8], x[8];
        ld8f(sT + i * kAS + j0, t8);
        ld8f(sBeta + j0, b8);
        if (a.T2) {
            const uint4 hi = pack8(t8);
            unpack8(hi, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = t8[e] - x[e];
            const size_t go = (size_t)crow * kC * kC + (size_t)i * kC + j0;
            *reinterpret_cast<uint4*>(a.T2 + go) = hi;
            *reinterpret_cast<uint4*>(a.Tlo + go) = pack8(x);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = t8[e] * b8[e];
        const uint4 pk = pack8(x);
        *reinterpret_cast<uint4*>(smem + J_TB + sw128_offset(i, j0)) = pk;
        *reinterpret_cast<uint4*>(smem + J_TB + sw128_offset(64 + i, j0)) = pk;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // W = (T beta) Khat into TMEM columns 0..127, U = (T beta) V into 128..255
    // (rows t in lanes 0..63, repeated in 64..127)
    if (tid == 0 && ok && wait_bar(bar_v, ph, 34)) {
        ++v_waited;
        tc_fence_after();
        const uint32_t id = idesc_bf16_f32(128, 128) | kBMajorMN;
        const uint32_t tb = smem_u32(smem + J_TB), kh = smem_u32(smem + J_G),
                       vt = smem_u32(smem + J_Q);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            mma_bf16(tmem + 0, sdesc_sw128(tb + kk * 32), sdesc_mn_sw128(kh + kk * 2048, 8192), id,
                     kk > 0);
            mma_bf16(tmem + 128, sdesc_sw128(tb + kk * 32), sdesc_mn_sw128(vt + kk * 2048, 8192),
                     id, kk > 0);
        }
        mma_commit(bar_w);
    }
    ok = ok && wait_bar_warp(bar_w, ph, 33);
    tc_fence_after();
    if (ok) {
        // quadrants 0, 1 read W rows into the g area (Khat's last reader was
        // the product), quadrants 2, 3 U rows into the q area (v's); warp
        // w / 4 takes the 64-column half
        const int isU = qd >> 1, cb = warp >> 2;
        float x0[32], x1[32];
        const uint32_t src = tmem + tlane + isU * 128 + cb * 64;
        tmem_ld32_nw(src, x0);
        tmem_ld32_nw(src + 32, x1);
        tmem_wait_ld_dep(x0);
        tmem_wait_ld_dep(x1);
        uint8_t* box = smem + (isU ? J_Q : J_G) + cb * 8192;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float e0[8], e1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                e0[i] = x0[8 * j + i];
                e1[i] = x1[8 * j + i];
            }
            *reinterpret_cast<uint4*>(box + sw128_offset(r, 8 * j)) = pack8(e0);
            *reinterpret_cast<uint4*>(box + sw128_offset(r, 32 + 8 * j)) = pack8(e1);
        }
        if (LO && isU) {
            __nv_bfloat16* ul = a.Ulo + (size_t)(row0 + r) * kD + cb * 64;
            store_lo32(ul, x0);
            store_lo32(ul + 32, x1);
        }
    }
    fence_async_smem();
    tc_fence_before();
    const bool all_ok = __syncthreads_and(ok);
    tc_fence_after();
    if (tid == 0 && all_ok) {
        tma_store_2d(&tm_w2, smem + J_G, 0, row0);
        tma_store_2d(&tm_w2, smem + J_G + 8192, 64, row0);
        tma_store_2d(&tm_u2, smem + J_Q, 0, row0);
        tma_store_2d(&tm_u2, smem + J_Q + 8192, 64, row0);
        bulk_commit_group();
        // the tiles (and the Aqk staging tile) are read before the next
        // chunk's loads overwrite them
        bulk_wait_read_all();
        if (next < total) issue_kqg(next);
    }
    if (!all_ok) break;
    }  // chunk loop
    // loads issued for chunks the loop did not reach (after an error) land
    // before shared memory is released, and every store has completed
    if (tid == 0) {
        for (; kqg_waited < kqg_issued; ++kqg_waited) wait_bar_drain(bar_kqg, kqg_waited & 1);
        for (; v_waited < v_issued; ++v_waited) wait_bar_drain(bar_v, v_waited & 1);
        bulk_wait_all();
        // every issued product completes before TMEM is released
        mma_commit(bar_fin);
        wait_bar_drain(bar_fin, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// Chunk-local backward on tensor cores (K = V = 128, chunk 64), one CTA of 512
// threads per (chunk, head); thread (c, R) = (tid % 128, tid / 128) owns key
// channel c of the 16-row block R, which is also TMEM lane c of its warp's
// quadrant.  With Y = diag(beta) (k o e^G):
//   P1  dT_raw = dW Y^T                 tcgen05, A = [dW; Y] (K-major, M=128)
//   P2  dKb'^T = dW^T T                 tcgen05, both operands MN-major
//   P3  Y2 = dT T^T, P4 dA = -mask(T^T Y2)   tcgen05 with every operand split
//       into bf16 hi + lo parts and three products (hi hi + hi lo + lo hi),
//       which keeps about 16 mantissa bits: T products need more than bf16
//   P5  row side, per block R: sum_j Right_R[j][c] [dA; dAqk][t][j]
//       (Right_R[j] = k_j e^{G_bR - G_j}, the intra kernel's operand)
//   P6  column side, per block pair (R, J<=R):
//       sum_{t in R} (beta k E)_t[c] dA[t][j] + (qs E)_t[c] dAqk[t][j]
//       combined with exp(G_bR - G_bJ) / E_j in the epilogue.
// The assembly then forms dk, dq, dG, dbeta and dg (reverse cumsum per
// channel in registers) exactly as the fp32 kernel does.
// ===========================================================================
constexpr uint32_t LB_K = 0, LB_Q = 16384, LB_G = 32768;     // TMA tiles, read up to the end
constexpr uint32_t LB_DWY = 49152;    // [dW; Y] 128 rows x 128, 2 k-blocks of 16 KB
// 81920 .. 90112: unused
constexpr uint32_t LB_DAQ = 90112;    // [dA_R; dAqk_R] rows 32R + 16s + u, 64 columns j
// T as [T_hi; T_lo]: bf16 [64 r][64 m] each, adjacent so that one N = 128
// operand covers both
constexpr uint32_t LB_T = 106496, LB_TLO = LB_T + 8192;
constexpr uint32_t LB_RIGHT = 122880; // Right_R tiles, 16(R+1) rows each
constexpr uint32_t LB_LCOL = 163840;  // [beta k E; qs E] rows 32R + 16s + u, 128 c
// dq, dk, dg staging tiles for their TMA stores ([64 t][128 c] bf16 as two
// 128B-swizzled 64-column boxes each), over Right and Lcol: free from the
// end of P5/P6 until the next chunk's operand build
constexpr uint32_t LB_STQ = LB_RIGHT, LB_STK = LB_RIGHT + 16384, LB_STG = LB_LCOL;
constexpr uint32_t LB_SMALL = 196608; // fp32 small arrays
constexpr uint32_t LB_F = LB_SMALL + 8192;   // F [6 block pairs][128] fp32
// LB_F + 3072 .. LB_SMALL + 16384: unused
constexpr uint32_t LB_DTV = LB_SMALL + 16384;  // dTv fp32 [64][64], 16-byte chunks XOR-swizzled
constexpr uint32_t LB_BAR = LB_DTV + 16384;
// After P1/P2 the [dW; Y] area holds the split P3/P4 operands.  P3's A has
// M = 128 rows of which only the first 64 matter: the hi tile's rows 64..127
// are the lo tile, the lo tile's rows 64..127 the Y2 hi tile.
constexpr uint32_t LB_DTH = LB_DWY, LB_DTL = LB_DWY + 8192;
constexpr uint32_t LB_Y2H = LB_DWY + 16384, LB_Y2L = LB_DWY + 24576;
constexpr uint32_t LOCAL_TC_SMEM = LB_BAR + 64 + 1024;
static_assert(LOCAL_TC_SMEM <= 232448, "local backward exceeds the per-CTA shared memory limit");
static_assert(LB_K % 1024 == 0 && LB_Q % 1024 == 0 && LB_G % 1024 == 0 && LB_DWY % 1024 == 0 &&
                  LB_T % 1024 == 0 && LB_TLO % 1024 == 0 && LB_DAQ % 1024 == 0 &&
                  LB_RIGHT % 1024 == 0 && LB_LCOL % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte aligned bases");
constexpr int kLocalTcThreads = 512;

__host__ __device__ constexpr uint32_t right_rel(int R) { return 2048u * (uint32_t)(R * (R + 1)); }
// fp32 dKb row r (512 bytes) in the assembly, staged in three freed areas
__host__ __device__ constexpr uint32_t lb_dkb_row(int r) {
    return r < 32 ? LB_DTV + 512u * r : r < 48 ? LB_T + 512u * (r - 32) : LB_TLO + 512u * (r - 48);
}

struct LocalTcArgs {
    int T, H, HV, NT, G, BH;
    int D;              // K of the tensors (64 or 128); the kernel works at 128
    float scale;
    int qkn;   // L2-normalise the q and k tiles first; dq, dk then go out as fp32
    const float *dQh, *dKb, *dTv, *dgam, *dbv;
    const __nv_bfloat16 *q, *k, *g, *beta;
    __nv_bfloat16 *dq, *dk, *dg, *dbeta;
    float *dqh, *dkh;
    const int* ctab;    // packed sequences: the chunk table, or null
};

// DW: K of the tensors (64 or 128), a compile-time constant (see grad_v).
// VL: packed sequences (a.ctab); a separate instantiation, so that the
// fixed-length one carries no row masks.
template <int DW, bool VL>
__global__ void __launch_bounds__(kLocalTcThreads, 1)
local_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_dw,    // dW bf16 [BH*T][128]
                    const __grid_constant__ CUtensorMap tm_t,     // T high part [BH*NT*64][64]
                    const __grid_constant__ CUtensorMap tm_tlo,   // T low part
                    const __grid_constant__ CUtensorMap tm_daq,   // dAqk bf16, 16-row boxes
                    const __grid_constant__ CUtensorMap tm_dqo,   // dq, dk, dg token tensors:
                    const __grid_constant__ CUtensorMap tm_dko,   // the outputs' TMA stores
                    const __grid_constant__ CUtensorMap tm_dgo,
                    LocalTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + LB_BAR);
    uint64_t* bar_m1 = bar_tma + 1;
    uint64_t* bar_m2 = bar_tma + 2;
    uint64_t* bar_m3 = bar_tma + 3;
    uint64_t* bar_m4 = bar_tma + 4;
    uint64_t* bar_g = bar_tma + 5;   // g tile (loaded apart from the others)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar_tma + 6);
    float* sBeta = reinterpret_cast<float*>(smem + LB_SMALL);   // [64]
    float* sDbp = sBeta + 64;                                   // [4 lane quadrants][64]
    float* sGtot = sDbp + 4 * 64;                               // [4][128]
    float* sGb = sGtot + 4 * kD;                                // [4][128]
    float* sLast = sGb + 4 * kD;                                // [4][128]
    float* sDtv = reinterpret_cast<float*>(smem + LB_DTV);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = tid & (kD - 1), R = tid >> 7;
    const uint32_t lane_off = (uint32_t)((c >> 5) * 32) << 16;
    const int total = a.BH * a.NT;   // chunks; CTA i takes chunks i, i + grid, ...

    // thread 0's counts of issued and consumed loads (every load is waited for
    // before the CTA exits), kept in shared memory so that they hold no
    // register in the other threads
    int* cnt = reinterpret_cast<int*>(sLast + 4 * kD);   // [main issued, g issued, main, g waited]
    int& main_issued = cnt[0];
    int& g_issued = cnt[1];
    int& main_waited = cnt[2];
    int& g_waited = cnt[3];
    // k, q tiles; dW into the top half of [dW; Y]; T (hi, lo) tiles; dAqk rows
    // into the rows 32R + 16 + u of [dA; dAqk]
    auto issue_main = [&](int ch) {
        const int nn = ch % a.NT, bb = ch / a.NT, hvv = bb % a.HV, hh = hvv / a.G;
        const int tr = tok_row(VL ? a.ctab : nullptr, bb / a.HV, a.T, nn), rw = bb * a.T + nn * kC, c64 = ch * kC;
        mbar_arrive_expect_tx(bar_tma, 2 * 16384 + 16384 + 2 * 8192 + 8192);
        tma_load_3d(smem + LB_K, &tm_k, bar_tma, 0, hh, tr);
        tma_load_3d(smem + LB_K + 8192, &tm_k, bar_tma, 64, hh, tr);
        tma_load_3d(smem + LB_Q, &tm_q, bar_tma, 0, hh, tr);
        tma_load_3d(smem + LB_Q + 8192, &tm_q, bar_tma, 64, hh, tr);
        tma_load_2d(smem + LB_DWY, &tm_dw, bar_tma, 0, rw);
        tma_load_2d(smem + LB_DWY + 16384, &tm_dw, bar_tma, 64, rw);
        tma_load_2d(smem + LB_T, &tm_t, bar_tma, 0, c64);
        tma_load_2d(smem + LB_TLO, &tm_tlo, bar_tma, 0, c64);
#pragma unroll
        for (int RR = 0; RR < 4; ++RR)
            tma_load_2d(smem + LB_DAQ + (32 * RR + 16) * 128, &tm_daq, bar_tma, 0, c64 + 16 * RR);
        ++main_issued;
    };
    auto issue_g = [&](int ch) {
        const int nn = ch % a.NT, bb = ch / a.NT, hvv = bb % a.HV;
        const int tr = tok_row(VL ? a.ctab : nullptr, bb / a.HV, a.T, nn);
        mbar_arrive_expect_tx(bar_g, 16384);
        tma_load_3d(smem + LB_G, &tm_g, bar_g, 0, hvv, tr);
        tma_load_3d(smem + LB_G + 8192, &tm_g, bar_g, 64, hvv, tr);
        ++g_issued;
    };
    // dTv (fp32) staged asynchronously by every thread; row i, 16-byte chunk
    // qd lands in chunk qd ^ (i & 7), so a thread reading its own row's chunks
    // meets no bank conflict within 8 lanes
    auto issue_dtv = [&](int ch) {
        const size_t cc = (size_t)ch * kC * kC;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int w = tid + e * kLocalTcThreads;
            const int i = w >> 4, qd = w & 15;
            cp_async16(sDtv + i * kC + ((qd ^ (i & 7)) << 2), a.dTv + cc + w * 4);
        }
        cp_async_commit();
    };
    auto load_beta = [&](int ch) {   // 0 past a packed sequence's end
        const int nn = ch % a.NT, bb = ch / a.NT;
        const int* ct = VL ? a.ctab : nullptr;
        return tid < tok_len(ct, nn)
                   ? __bfloat162float(a.beta[((size_t)tok_row(ct, bb / a.HV, a.T, nn) + tid) * a.HV +
                                             bb % a.HV])
                   : 0.f;
    };

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_m1, 1);
        mbar_init(bar_m2, 1);
        mbar_init(bar_m3, 1);
        mbar_init(bar_m4, 1);
        mbar_init(bar_g, 1);
        fence_mbar_init();
        cnt[0] = cnt[1] = cnt[2] = cnt[3] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if ((int)blockIdx.x < total) {
        if (tid == 0) {
            issue_g(blockIdx.x);
            issue_main(blockIdx.x);
        }
        issue_dtv(blockIdx.x);
    }
    float beta_next = (tid < kC && (int)blockIdx.x < total) ? load_beta(blockIdx.x) : 0.f;
    bool ok = true;

#pragma unroll 1
    for (int it = 0, chunk = blockIdx.x; chunk < total; ++it, chunk += gridDim.x) {
    const uint32_t ph = it & 1;
    const int next = chunk + gridDim.x;
    const int n = chunk % a.NT, bh = chunk / a.NT;
    const int b = bh / a.HV, hv = bh % a.HV;
    const int trow = tok_row(VL ? a.ctab : nullptr, b, a.T, n);
    const int len = tok_len(VL ? a.ctab : nullptr, n);   // valid rows (a partial chunk of a packed batch)
    const size_t row0 = (size_t)bh * a.T + (size_t)n * kC;
    if (tid < kC) {
        sBeta[tid] = tid < len ? beta_next : 0.f;        // read after later barriers
        if (next < total) beta_next = load_beta(next);   // in flight meanwhile
    }
    {
        const bool got = wait_bar_warp(bar_g, ph, 46);
        if (got && tid == 0) ++g_waited;
        ok = ok && got;
    }
    if (len < kC) {   // rows past the end of a packed sequence: g = 0
        zero_tile_rows(smem + LB_G, len, tid, kLocalTcThreads);
        __syncthreads();
    }

    const uint32_t kbo = (c >> 6) * 8192, cc = c & 63;
    auto ldt = [&](uint32_t tile, int r) {
        return __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16*>(smem + tile + kbo + sw128_offset(r, cc)));
    };
    // ---- cumsum (thread (c, R): rows 16R..16R+15 of channel c); the gate mask
    // [g >= -5] of the rows is kept for dg, so the g tile is free afterwards ----
    float G[16];
    uint32_t gmask = 0;
    {
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const float gv = ldt(LB_G, 16 * R + u);
            gmask |= (gv >= kGateFloor ? 1u : 0u) << u;
            acc += fmaxf(gv, kGateFloor);
            G[u] = acc;
        }
        sGtot[R * kD + c] = acc;
    }
    // the previous chunk's output stores have read the staging tiles before
    // the operand build below rewrites them
    if (!VL && tid == 0) bulk_wait_read_all();
    __syncthreads();
    if (tid == 0 && next < total) issue_g(next);   // the next chunk's g tile
    float off = 0.f, Glast = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float t = sGtot[p * kD + c];
        if (p < R) off += t;
        Glast += t;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) G[u] += off;
    sGb[R * kD + c] = G[0];
    __syncthreads();
    float Gb[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) Gb[p] = sGb[p * kD + c];
    const float eGbR = __expf(Gb[R]), eLbR = __expf(Glast - Gb[R]);
    // F(R, Rd) = exp(G_b(Rd) - G_b(R)) for the later blocks Rd, per channel: the
    // factors of the Right copies below
    {
        float* sF = reinterpret_cast<float*>(smem + LB_F);
#pragma unroll
        for (int Rd = 1; Rd < 4; ++Rd)
            if (Rd > R) sF[f_slot(R, Rd) * kD + c] = __expf(Gb[Rd] - Gb[R]);
    }
    {
        const bool got = wait_bar_warp(bar_tma, ph, 41);
        if (got && tid == 0) ++main_waited;
        ok = ok && got;
    }
    if (len < kC) {   // and q = k = 0 there
        zero_tile_rows(smem + LB_K, len, tid, kLocalTcThreads);
        zero_tile_rows(smem + LB_Q, len, tid, kLocalTcThreads);
        __syncthreads();
    }
    if (a.qkn) {
        l2norm_tile_rows(smem + LB_K, tid, kLocalTcThreads);
        l2norm_tile_rows(smem + LB_Q, tid, kLocalTcThreads);
        __syncthreads();
    }

    // ---- build bf16 operands: Y, Right_R (own block; the copies for later
    // blocks follow while P1/P2 run), Lcol.  The G values of a quad of lanes
    // (channels cq..cq+3) are first transposed within the quad, so that lane
    // s of the quad owns rows 16R + 4s .. + 3 of all four channels: every
    // load and store then moves four channels (8 bytes) at once. ----
    {
        const int s4 = lane & 3, cq = c - s4;
        // GT[4 i + j]: channel cq + i, row 16R + 4 s4 + j.  A 4 x 4 transpose of
        // 4-row blocks across the quad: at stage m, of each block pair
        // (b, b ^ m) a lane keeps the one on its side of bit m and receives the
        // partner's other one.
        float GT[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) GT[u] = G[u];
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
            const bool up = (s4 & m) != 0;
#pragma unroll
            for (int b0 = 0; b0 < 4; ++b0) {
                if (b0 & m) continue;
                const int b1 = b0 ^ m;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float send = up ? GT[4 * b0 + k] : GT[4 * b1 + k];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, m);
                    if (up)
                        GT[4 * b0 + k] = recv;
                    else
                        GT[4 * b1 + k] = recv;
                }
            }
        }
        const float4 gb4 = *reinterpret_cast<const float4*>(sGb + R * kD + cq);
        const float gbq[4] = {gb4.x, gb4.y, gb4.z, gb4.w};
        float egb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) egb[i] = __expf(gbq[i]);
        const float4 bt4 = *reinterpret_cast<const float4*>(sBeta + 16 * R + 4 * s4);
        const float btq[4] = {bt4.x, bt4.y, bt4.z, bt4.w};
        const uint32_t kbq = (cq >> 6) * 8192, cb16 = (cq >> 6) * 16384, ccq = cq & 63;
        const uint32_t rbase = LB_RIGHT + right_rel(R) + (cq >> 6) * (16u * (R + 1) * 128u);
        auto st4 = [&](uint32_t off, const float (&x)[4]) {
            *reinterpret_cast<uint2*>(smem + off) =
                make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
        };
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int u = 4 * s4 + j, r = 16 * R + u;
            const uint32_t so = sw128_offset(r, ccq);
            const uint2 k2 = *reinterpret_cast<const uint2*>(smem + LB_K + kbq + so);
            const uint2 q2 = *reinterpret_cast<const uint2*>(smem + LB_Q + kbq + so);
            const float2 k01 = unpack_bf16(k2.x), k23 = unpack_bf16(k2.y);
            const float2 q01 = unpack_bf16(q2.x), q23 = unpack_bf16(q2.y);
            const float kv[4] = {k01.x, k01.y, k23.x, k23.y};
            const float qv[4] = {q01.x, q01.y, q23.x, q23.y};
            float y[4], rt[4], l1[4], l2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float E = __expf(GT[4 * i + j] - gbq[i]);
                const float Einv = __expf(gbq[i] - GT[4 * i + j]);
                l1[i] = btq[j] * kv[i] * E;             // beta k E
                y[i] = l1[i] * egb[i];                  // Y = beta k exp(G)
                rt[i] = kv[i] * Einv;                   // Right_R
                l2[i] = a.scale * qv[i] * E;            // qs E
            }
            st4(LB_DWY + cb16 + sw128_offset(64 + r, ccq), y);   // Y rows of [dW; Y]
            st4(rbase + so, rt);
            st4(LB_LCOL + cb16 + sw128_offset(32 * R + u, ccq), l1);
            st4(LB_LCOL + cb16 + sw128_offset(32 * R + 16 + u, ccq), l2);
        }
    }
    cp_async_wait_all16();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- P1, P2 ----
    if (tid == 0 && ok) {
        const uint32_t dwy = smem_u32(smem + LB_DWY), tt = smem_u32(smem + LB_T);
        const uint32_t id64 = idesc_bf16_f32(128, 64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem + 0, sdesc_sw128(dwy + ko), sdesc_sw128(dwy + 8192 + ko), id64, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 64, sdesc_mn_sw128(dwy + kk * 2048, 16384),
                     sdesc_mn_sw128(tt + kk * 2048, 8192), id64 | kAMajorMN | kBMajorMN, kk > 0);
        mma_commit(bar_m1);
    }
    // Right_Rr rows of block R for Rr > R: Right_R scaled by F(R, Rr), 16-byte
    // units (6 block pairs x 16 rows x 16 chunks) spread over all threads
    // while P1/P2 run; pair pr is F's slot
#pragma unroll 1
    for (int e = 0; e < 3; ++e) {
        const int w = tid + e * kLocalTcThreads, pr = w >> 8, rem = w & 255;
        const int Rs = pr < 3 ? 0 : pr < 5 ? 1 : 2;
        const int Rd = pr < 3 ? pr + 1 : pr < 5 ? pr - 1 : 3;
        const int r = 16 * Rs + (rem >> 4), oct = rem & 15, kb = oct >> 3, ch = oct & 7;
        const uint32_t co = (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
        float f8[8], x[8];
        ld8f(reinterpret_cast<const float*>(smem + LB_F) + pr * kD + oct * 8, f8);
        unpack8(*reinterpret_cast<const uint4*>(smem + LB_RIGHT + right_rel(Rs) +
                                                 kb * (16u * (Rs + 1) * 128u) + co), x);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= f8[i];
        *reinterpret_cast<uint4*>(smem + LB_RIGHT + right_rel(Rd) + kb * (16u * (Rd + 1) * 128u) +
                                  co) = pack8(x);
    }
    ok = ok && wait_bar_warp(bar_m1, ph, 42);
    tc_fence_after();
    // Epilogues below run in the warps of TMEM quadrants 0 and 1 (c < 64):
    // thread (c, R) owns row c of a 64 x 64 result, columns 16R..16R+15,
    // written as two 16-byte units per tile (a warp's 32 rows then fill all
    // banks; single bf16 stores down a column would conflict 4 ways).
    // split8 stores x as bf16 hi + lo parts at byte offset off of two tiles.
    auto split8 = [&](uint32_t hi, uint32_t lo, uint32_t off, const float (&x)[8]) {
        float h[8], l[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            h[e] = __bfloat162float(__float2bfloat16_rn(x[e]));
            l[e] = x[e] - h[e];
        }
        *reinterpret_cast<uint4*>(smem + hi + off) = pack8(h);
        *reinterpret_cast<uint4*>(smem + lo + off) = pack8(l);
    };
    // ---- dT = mask_strict(beta_m dTv + dW Y^T), split hi + lo ----
    if (ok && c < kC) {
        float r16[16];
        tmem_ld16(tmem + lane_off + 16 * R, r16);
        const int i = c;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x8[8];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int q4 = 4 * R + 2 * hh + x;
                const float4 t4 =
                    *reinterpret_cast<const float4*>(sDtv + i * kC + ((q4 ^ (i & 7)) << 2));
                const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 4 * q4 + e;
                    x8[4 * x + e] = m < i ? sBeta[m] * tv[e] + r16[8 * hh + 4 * x + e] : 0.f;
                }
            }
            split8(LB_DTH, LB_DTL, sw128_offset(i, 16 * R + 8 * hh), x8);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- P3: Y2 = dT T^T.  dT_hi [T_hi; T_lo]^T (N = 128) puts hi.hi in TMEM
    // columns 128..191 and hi.lo in 192..255; dT_lo T_hi^T adds onto 128..191 ----
    if (tid == 0 && ok) {
        const uint32_t dth = smem_u32(smem + LB_DTH), dtl = smem_u32(smem + LB_DTL);
        const uint32_t th = smem_u32(smem + LB_T);
        const uint32_t id64 = idesc_bf16_f32(128, 64), id128 = idesc_bf16_f32(128, 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 128, sdesc_sw128(dth + kk * 32), sdesc_sw128(th + kk * 32), id128,
                     kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 128, sdesc_sw128(dtl + kk * 32), sdesc_sw128(th + kk * 32), id64, 1);
        mma_commit(bar_m3);
    }
    ok = ok && wait_bar_warp(bar_m3, ph, 44);
    tc_fence_after();
    if (ok && c < kC) {
        float r16[16], s16[16];
        tmem_ld16(tmem + lane_off + 128 + 16 * R, r16);
        tmem_ld16(tmem + lane_off + 192 + 16 * R, s16);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x8[e] = r16[8 * hh + e] + s16[8 * hh + e];
            split8(LB_Y2H, LB_Y2L, sw128_offset(c, 16 * R + 8 * hh), x8);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- P4: T^T Y2, T and Y2 read MN-major.  T_hi^T [Y2_hi | Y2_lo] (N = 128
    // over the adjacent Y2 tiles) puts hi.hi in TMEM columns 256..319 and hi.lo
    // in 320..383; T_lo^T Y2_hi adds onto 256..319.  A spans M = 128: its
    // second MN block (+8192 B) is don't-care data ----
    if (tid == 0 && ok) {
        const uint32_t th = smem_u32(smem + LB_T), tl = smem_u32(smem + LB_TLO);
        const uint32_t yh = smem_u32(smem + LB_Y2H);
        const uint32_t id64 = idesc_bf16_f32(128, 64) | kAMajorMN | kBMajorMN;
        const uint32_t id128 = idesc_bf16_f32(128, 128) | kAMajorMN | kBMajorMN;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 256, sdesc_mn_sw128(th + kk * 2048, 8192),
                     sdesc_mn_sw128(yh + kk * 2048, 8192), id128, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 256, sdesc_mn_sw128(tl + kk * 2048, 8192),
                     sdesc_mn_sw128(yh + kk * 2048, 8192), id64, 1);
        mma_commit(bar_m4);
    }
    ok = ok && wait_bar_warp(bar_m4, ph, 45);
    tc_fence_after();
    // stage the assembly's fp32 inputs dQh (into the [dW; Y] area) and dKb
    // (rows 0..31 into the dTv area, 32..47 into T, 48..63 into T's low part):
    // all of them were last read by P4
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int ch = tid + e * kLocalTcThreads, r = ch >> 5, c4 = (ch & 31) * 4;
        cp_async16(smem + LB_DWY + r * 512 + c4 * 4, a.dQh + (row0 + r) * kD + c4);
        cp_async16(smem + lb_dkb_row(r) + c4 * 4, a.dKb + (row0 + r) * kD + c4);
    }
    cp_async_commit();
    // dA = -mask_strict(T^T Y2) (bf16) into the row-side and column-side B tiles
    if (ok && c < kC) {
        float r16[16], s16[16];
        tmem_ld16(tmem + lane_off + 256 + 16 * R, r16);
        tmem_ld16(tmem + lane_off + 320 + 16 * R, s16);
        const int i = c, t2 = 32 * (i >> 4) + (i & 15);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 16 * R + 8 * hh + e;
                x8[e] = j < i ? -(r16[8 * hh + e] + s16[8 * hh + e]) : 0.f;
            }
            *reinterpret_cast<uint4*>(smem + LB_DAQ + sw128_offset(t2, 16 * R + 8 * hh)) = pack8(x8);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- P5 (row side), P6 (column side) ----
    if (tid == 0 && ok) {
        const uint32_t daq = smem_u32(smem + LB_DAQ);
        const uint32_t right = smem_u32(smem + LB_RIGHT), lcol = smem_u32(smem + LB_LCOL);
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) {
            const uint32_t id = idesc_bf16_f32(128, 32) | kAMajorMN;
            for (int kk = 0; kk <= RR; ++kk)
                mma_bf16(tmem + 128 + 32 * RR,
                         sdesc_mn_sw128(right + right_rel(RR) + kk * 2048, 2048u * (RR + 1)),
                         sdesc_sw128(daq + 4096u * RR + kk * 32), id, kk > 0);
        }
        // one MMA per block R covers the pairs (R, J <= R): B is [dA; dAqk]
        // read MN-major (N = its 64 columns j, K = its rows 32R..32R+31), so
        // pair (R, J) lands in TMEM columns 256 + 64 R + 16 J (J > R unused)
#pragma unroll
        for (int RR = 0; RR < 4; ++RR) {
            const uint32_t id = idesc_bf16_f32(128, 64) | kAMajorMN | kBMajorMN;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                mma_bf16(tmem + 256 + 64 * RR,
                         sdesc_mn_sw128(lcol + 4096u * RR + kk * 2048, 16384),
                         sdesc_mn_sw128(daq + 4096u * RR + kk * 2048, 8192), id, kk > 0);
        }
        mma_commit(bar_m2);
    }
    ok = ok && wait_bar_warp(bar_m2, ph, 43);
    tc_fence_after();
    cp_async_wait_all16();
    __syncthreads();

    // ---- assembly: thread (c, R) for rows t = 16R + u ----
    float dG[16], dbps[16];
    float lastp = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) dbps[u] = 0.f;
    if (ok) {
        float dkb[16], cAQ[16], sAQ[32];
        tmem_ld16(tmem + lane_off + 64 + 16 * R, dkb);          // d(beta khat) for t in R
        tmem_ld32(tmem + lane_off + 128 + 32 * R, sAQ);         // sA raw | sQ raw
#pragma unroll
        for (int u = 0; u < 16; ++u) cAQ[u] = 0.f;
        for (int Rp = R; Rp < 4; ++Rp) {
            float d6[16];
            tmem_ld16(tmem + lane_off + 256 + 64 * Rp + 16 * R, d6);
            const float f = Rp > R ? __expf(Gb[Rp] - Gb[R]) : 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) cAQ[u] += f * d6[u];
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * R + u;
            const float E = __expf(G[u] - Gb[R]);
            const float Einv = __expf(Gb[R] - G[u]);
            const float eG = eGbR * E, eL = eLbR * Einv;
            const float kr = ldt(LB_K, t);
            const float qr = a.scale * ldt(LB_Q, t);
            const float br = sBeta[t];
            const float dKbeta = dkb[u];
            const float dQh = *reinterpret_cast<const float*>(smem + LB_DWY + t * 512 + c * 4);
            const float dKb = *reinterpret_cast<const float*>(smem + lb_dkb_row(t) + c * 4);
            const float sa = sAQ[u] * E, sq = sAQ[16 + u] * E, caq = cAQ[u] * Einv;
            // with p = dKbeta eG + sa (the factor beta multiplies) and l = dKb eL:
            // dk = beta p + l + caq, dqs = dQh eG + sq,
            // dG = k (beta p - l - caq) + qs dqs, dbeta partial = k p
            const float pb = fmaf(dKbeta, eG, sa), l = dKb * eL, bp = br * pb;
            const float dkv = bp + l + caq;
            const float dqs = fmaf(dQh, eG, sq);
            dG[u] = fmaf(qr, dqs, kr * (bp - l - caq));
            lastp = fmaf(kr, l, lastp);
            dbps[u] = kr * pb;
            const size_t io = (((size_t)trow + t) * a.HV + hv) * DW + c;
            if ((DW < kD && c >= DW) || t >= len) {
                // a key channel past the tensors' width (zero-filled), or a
                // row past a packed sequence's end: not written
            } else if (a.G == 1 && !a.qkn) {
                if (!VL) {   // into the staging tiles, for one TMA store each
                    const uint32_t so = (uint32_t)(c >> 6) * 8192 + sw128_offset(t, c & 63);
                    *reinterpret_cast<__nv_bfloat16*>(smem + LB_STQ + so) =
                        __float2bfloat16_rn(a.scale * dqs);
                    *reinterpret_cast<__nv_bfloat16*>(smem + LB_STK + so) = __float2bfloat16_rn(dkv);
                } else {
                    a.dq[io] = __float2bfloat16_rn(a.scale * dqs);
                    a.dk[io] = __float2bfloat16_rn(dkv);
                }
            } else {
                a.dqh[io] = a.scale * dqs;
                a.dkh[io] = dkv;
            }
        }
    } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) dG[u] = 0.f;
    }
    // the tail's global inputs, in flight while the partial sums are formed
    const float dgam_c = a.dgam[((size_t)bh * a.NT + n) * kD + c];
    const float dbv_t = tid < kC ? a.dbv[row0 + tid] : 0.f;
    // dbeta partials of rows 16R..16R+15 over this warp's 32 channels: lane
    // pair (2u, 2u+1) ends with row 16R + u
    {
        const float tot = warp_sum_scatter<16>(dbps);
        if (!(lane & 1)) sDbp[(warp & 3) * 64 + 16 * R + (lane >> 1)] = tot;
    }
    // block sums of dG and the last-row partials, for the reverse cumsum
    float bsum = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) bsum += dG[u];
    sGtot[R * kD + c] = bsum;
    sLast[R * kD + c] = lastp;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // k, q, [dW; Y], T, [dA; dAqk] and the staging areas have been read: the
    // next chunk's loads start while this chunk's tail runs
    if (next < total && ok) {
        if (tid == 0) issue_main(next);
        issue_dtv(next);
    }
    if (!VL && tid == 0 && ok && a.G == 1 && !a.qkn) {   // dq, dk (key head = value head)
        tma_store_3d(&tm_dqo, smem + LB_STQ, 0, hv, trow);
        tma_store_3d(&tm_dko, smem + LB_STK, 0, hv, trow);
        if (DW > 64) {
            tma_store_3d(&tm_dqo, smem + LB_STQ + 8192, 64, hv, trow);
            tma_store_3d(&tm_dko, smem + LB_STK + 8192, 64, hv, trow);
        }
        bulk_commit_group();
    }
    {
        // dG_last += sum_r dKb_r Kb_r + dgam gam; it enters every row's suffix sum
        float extra = dgam_c * __expf(Glast);
#pragma unroll
        for (int p = 0; p < 4; ++p) extra += sLast[p * kD + c];
        float run = extra;
        for (int p = R + 1; p < 4; ++p) run += sGtot[p * kD + c];
#pragma unroll
        for (int u = 15; u >= 0; --u) {
            run += dG[u];
            const int t = 16 * R + u;
            const size_t ig = (((size_t)trow + t) * a.HV + hv) * DW + c;
            if ((DW == kD || c < DW) && t < len) {
                const __nv_bfloat16 x = __float2bfloat16_rn((gmask >> u) & 1u ? run : 0.f);
                if (!VL)
                    *reinterpret_cast<__nv_bfloat16*>(smem + LB_STG + (uint32_t)(c >> 6) * 8192 +
                                                      sw128_offset(t, c & 63)) = x;
                else
                    a.dg[ig] = x;
            }
        }
    }
    if (tid < len)
        a.dbeta[((size_t)trow + tid) * a.HV + hv] =
            __float2bfloat16_rn((sDbp[tid] + sDbp[64 + tid]) + (sDbp[128 + tid] + sDbp[192 + tid]) +
                                dbv_t);
    // partial sums, beta and TMEM are reused by the next chunk
    fence_async_smem();
    tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    if (!VL && tid == 0) {   // dg from its staging tile
        tma_store_3d(&tm_dgo, smem + LB_STG, 0, hv, trow);
        if (DW > 64) tma_store_3d(&tm_dgo, smem + LB_STG + 8192, 64, hv, trow);
        bulk_commit_group();
    }
    }  // chunk loop
    // loads issued for chunks the loop did not reach (after an error) land
    // before shared memory is released, and the output stores complete
    if (tid == 0) bulk_wait_all();
    cp_async_wait_all16();
    if (tid == 0) {
        for (; main_waited < main_issued; ++main_waited) wait_bar_drain(bar_tma, main_waited & 1);
        for (; g_waited < g_issued; ++g_waited) wait_bar_drain(bar_g, g_waited & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- host: tensor maps ----
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encoder() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// SMs of the current device (cached per device), for persistent grids.
int sm_count() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

// A second stream per device, created on first use: the recomputing backward
// runs its reverse state pass there, beside the forward state pass.
cudaStream_t aux_stream() {
    static std::mutex mu;
    static cudaStream_t per_dev[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!per_dev[dev] && cudaStreamCreateWithFlags(&per_dev[dev], cudaStreamNonBlocking) != cudaSuccess)
        per_dev[dev] = nullptr;
    return per_dev[dev];
}

// 2-D bf16 map over a row-major [rows][cols] array with a box of
// box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows, bool swizzle128) {
    EncodeFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 2-D fp32 map over a row-major [rows][cols] array, no swizzle (a plain
// row-major shared-memory box of box_cols x box_rows).
bool make_map_f32(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows) {
    EncodeFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 3-D bf16 map over a token tensor [B*T][heads][128] (a per-head tile of 64
// tokens is a box {64 columns, 1 head, 64 tokens}), 128B swizzle.
// The row width D (64 or 128) is the tensor's own: with D = 64 the box at
// column 64 lies wholly past the row, so TMA loads fill it with zeros and
// stores skip it, and the 128-wide kernels see zero channels there.
bool make_map_tok(CUtensorMap* m, const void* ptr, uint64_t BT, uint64_t heads, uint64_t D) {
    EncodeFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {D, heads, BT};
    cuuint64_t strides[2] = {D * 2, heads * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

struct TcWs {
    char* simt;  // SIMT workspace (fp32 quantities)
    __nv_bfloat16 *W2, *Q2, *U2, *Kb2, *Aqk2, *T2, *Tlo2;  // chain operands, T (hi, lo)
    __nv_bfloat16 *h2, *d2, *dh2, *dd2;              // backward only
    // low parts of the two-term split (backward with an upstream final-state
    // gradient): U, Kb, delta^T, dS^T; dhlo takes the space of U2 and Ulo,
    // which the recompute has read before the reverse pass writes it
    __nv_bfloat16 *Ulo, *Kblo, *d2lo, *dhlo;
    float *sbuf, *zbuf, *mbuf, *ident;               // segmented forward scan (plain forward)
};

// Segments of the plain forward's state pass (0: one run over all chunks).
// Its first launch holds BH (2P - 3) CTAs of one SM each and should fit one
// wave; P >= 3, at least 16 chunks per segment.  Cutting the sequence only
// pays when few heads leave most SMs idle during a long state pass.
int chain_segments(const kda_dims& d) {
    const int BH = d.B * d.HV, NT = d.T / kC;
    if (BH <= 0 || NT < 48) return 0;
    int P = (sm_count() / BH + 3) / 2;
    P = std::min(P, 8);
    P = std::min(P, NT / 16);
    return P >= 3 ? P : 0;
}

// The tensor-core kernels work at K = V = 128 whatever the tensors' width
// (64 or 128): the fp32 arrays they share with the SIMT carve are laid out
// at that width.
kda_dims tc_wide(const kda_dims& d) {
    kda_dims p = d;
    p.K = p.V = kD;
    return p;
}

// A packed variable-length batch: the chunk table and each sequence's first
// chunk slot (in the workspace), the sequence count and the real token count.
// The kernels then see B = 1 and T = the padded slot count times 64 (the
// workspace arrays' row count); the token tensors have Ttok rows.
struct TcVl {
    const int *ctab, *sfirst;
    int nseq, Ttok;
};
inline uint64_t tok_rows(const kda_dims& d, const TcVl* vl) {
    return vl ? (uint64_t)vl->Ttok : (uint64_t)d.B * d.T;
}

size_t tc_carve(const kda_dims& d, int for_bwd, char* base, TcWs* w) {
    const size_t BH = (size_t)d.B * d.HV, T = d.T, NT = d.T / kC;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    auto bf = [&](size_t elems) { return reinterpret_cast<__nv_bfloat16*>(take(elems * 2)); };
    TcWs x{};
    x.simt = take(simt_workspace_bytes(tc_wide(d), for_bwd));
    x.W2 = bf(BH * T * kD);
    x.Q2 = bf(BH * T * kD);
    x.U2 = bf(BH * T * kD);
    if (for_bwd) {
        x.Ulo = bf(BH * T * kD);   // directly after U2: [BH][NT][V][K] fits both
        x.dhlo = x.U2;
    }
    x.Kb2 = bf(BH * T * kD);
    x.Aqk2 = bf(BH * NT * kC * kC);
    x.T2 = bf(BH * NT * kC * kC);
    x.Tlo2 = bf(BH * NT * kC * kC);
    if (for_bwd) {
        x.h2 = bf(BH * NT * kD * kD);
        x.d2 = bf(BH * T * kD);
        x.dh2 = bf(BH * NT * kD * kD);
        x.dd2 = bf(BH * T * kD);
        x.Kblo = bf(BH * T * kD);
        x.d2lo = bf(BH * NT * kD * kC);
    } else if (const int P = chain_segments(d)) {
        const size_t st = (size_t)d.K * d.V * sizeof(float);
        auto f32 = [&](size_t bytes) { return reinterpret_cast<float*>(take(bytes)); };
        x.sbuf = f32(BH * P * st);
        x.zbuf = f32(BH * P * st);
        x.mbuf = f32(BH * P * st);
        x.ident = f32(st);
    }
    if (w) *w = x;
    return off;
}

// Intra-chunk quantities on tensor cores, stored by TMA into the operand
// arrays (and gam, and T when kept, into the arrays the backward reads).
// keep_T: also write T as bf16 high and low parts (the backward needs them;
// the plain forward does not).
kda_status run_intra_tc(const kda_dims& d, const TcWs& w, const void* q, const void* k,
                        const void* v, const void* g, const void* beta, bool keep_T,
                        cudaStream_t s, float** gam_out, __nv_bfloat16* ulo = nullptr,
                        __nv_bfloat16* kblo = nullptr, const TcVl* vl = nullptr) {
    SimtWsPtrs p;
    simt_ws_ptrs(tc_wide(d), 0, w.simt, &p);
    const int BH = d.B * d.HV, NT = d.T / kC;
    const uint64_t BT = tok_rows(d, vl);
    const uint64_t rows = (uint64_t)BH * d.T;
    CUtensorMap mk, mq, mg, mv, mw2, mq2, mu2, mkb2, ma2;
    if (!make_map_tok(&mk, k, BT, d.H, d.K) || !make_map_tok(&mq, q, BT, d.H, d.K) ||
        !make_map_tok(&mg, g, BT, d.HV, d.K) || !make_map_tok(&mv, v, BT, d.HV, d.V) ||
        !make_map(&mw2, w.W2, rows, kD, 64, 64, true) ||
        !make_map(&mq2, w.Q2, rows, kD, 64, 64, true) ||
        !make_map(&mu2, w.U2, rows, kD, 64, 64, true) ||
        !make_map(&mkb2, w.Kb2, rows, kD, 64, 64, true) ||
        !make_map(&ma2, w.Aqk2, (uint64_t)BH * NT * kC, kC, 64, 64, true))
        return KDA_ERR_CUDA;
    IntraArgs a;
    a.T = d.T;
    a.H = d.H;
    a.HV = d.HV;
    a.NT = NT;
    a.BH = BH;
    a.D = d.K;
    a.scale = d.scale;
    a.qkn = d.qk_l2norm != 0;
    a.beta = static_cast<const __nv_bfloat16*>(beta);
    a.T2 = keep_T ? w.T2 : nullptr;
    a.Tlo = keep_T ? w.Tlo2 : nullptr;
    a.Ulo = ulo;
    a.Kblo = kblo;
    a.gam = p.gam;
    a.ctab = vl ? vl->ctab : nullptr;
    if ((ulo == nullptr) != (kblo == nullptr)) return KDA_ERR_INVALID_ARG;
    auto kern = vl ? (ulo ? intra_tc_kernel<true, true> : intra_tc_kernel<false, true>)
                   : (ulo ? intra_tc_kernel<true, false> : intra_tc_kernel<false, false>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)INTRA_SMEM) != cudaSuccess)
        return KDA_ERR_CUDA;
    {
        TimedLaunch tl("tc_intra", s);
        // persistent: two CTAs per SM walk the chunks
        const int grid = std::min(BH * NT, 2 * sm_count());
        kern<<<grid, kIntraThreads, INTRA_SMEM, s>>>(mk, mq, mg, mv, mw2, mq2, mu2, mkb2, ma2, a);
    }
    *gam_out = p.gam;
    return launch_status();
}

kda_status run_local_bwd_tc(const kda_dims& d, const TcWs& w, const SimtWsPtrs& p,
                            const void* q, const void* k, const void* g, const void* beta,
                            void* dq, void* dk, void* dg, void* dbeta, cudaStream_t s,
                            const TcVl* vl = nullptr) {
    const uint64_t BT = tok_rows(d, vl);
    const uint64_t rows = (uint64_t)d.B * d.HV * d.T;  // [BH*T] and [BH*NT*64] alike
    CUtensorMap mk, mq, mg, mdw, mt, mtl, mda;
    if (!make_map_tok(&mk, k, BT, d.H, d.K) || !make_map_tok(&mq, q, BT, d.H, d.K) ||
        !make_map_tok(&mg, g, BT, d.HV, d.K) || !make_map(&mdw, p.dWm, rows, kD, 64, 64, true) ||
        !make_map(&mt, w.T2, rows, kC, 64, 64, true) ||
        !make_map(&mtl, w.Tlo2, rows, kC, 64, 64, true) ||
        !make_map(&mda, p.dAqk, rows, kC, 64, 16, true))
        return KDA_ERR_CUDA;
    CUtensorMap mdqo, mdko, mdgo;   // the outputs (used by the fixed-length kernel)
    if (!make_map_tok(&mdqo, dq, BT, d.H, d.K) || !make_map_tok(&mdko, dk, BT, d.H, d.K) ||
        !make_map_tok(&mdgo, dg, BT, d.HV, d.K))
        return KDA_ERR_CUDA;
    LocalTcArgs a;
    a.T = d.T;
    a.H = d.H;
    a.HV = d.HV;
    a.NT = d.T / kC;
    a.G = d.HV / d.H;
    a.BH = d.B * d.HV;
    a.D = d.K;
    a.scale = d.scale;
    a.qkn = d.qk_l2norm != 0;
    a.dQh = p.dQh;
    a.dKb = p.dKb;
    a.dTv = p.dTv;
    a.dgam = p.dgam;
    a.dbv = p.dbv;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.g = static_cast<const __nv_bfloat16*>(g);
    a.beta = static_cast<const __nv_bfloat16*>(beta);
    a.dq = static_cast<__nv_bfloat16*>(dq);
    a.dk = static_cast<__nv_bfloat16*>(dk);
    a.dg = static_cast<__nv_bfloat16*>(dg);
    a.dbeta = static_cast<__nv_bfloat16*>(dbeta);
    a.dqh = p.dqh;
    a.dkh = p.dkh;
    a.ctab = vl ? vl->ctab : nullptr;
    auto kern = d.K == kD ? (vl ? local_bwd_tc_kernel<kD, true> : local_bwd_tc_kernel<kD, false>)
                          : (vl ? local_bwd_tc_kernel<64, true> : local_bwd_tc_kernel<64, false>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)LOCAL_TC_SMEM) != cudaSuccess)
        return KDA_ERR_CUDA;
    {
        TimedLaunch tl("tc_local_bwd", s);
        // persistent: one CTA per SM walks the chunks
        kern<<<std::min(a.BH * a.NT, sm_count()), kLocalTcThreads, LOCAL_TC_SMEM, s>>>(
            mk, mq, mg, mdw, mt, mtl, mda, mdqo, mdko, mdgo, a);
    }
    return launch_status();
}

// nseg >= 3: the plain forward as a segmented scan (three launches and a
// combine step; see ChainArgs), with its buffers in w.
kda_status run_chain_fwd(const kda_dims& d, const TcWs& w, const float* gam, const float* h0,
                         void* o, float* ht, __nv_bfloat16* h_out, __nv_bfloat16* delta_out,
                         cudaStream_t s, int nseg = 0, const __nv_bfloat16* u_lo = nullptr,
                         __nv_bfloat16* delta_lo = nullptr, const TcVl* vl = nullptr) {
    const int BH = d.B * d.HV, NT = d.T / kC;
    // one CTA per (b, hv), or per (sequence, hv) of a packed batch
    const int ctas = vl ? vl->nseq * d.HV : BH;
    CUtensorMap mw, mq, mk, ma, mu;
    const uint64_t rows = (uint64_t)BH * d.T;
    if (!make_map(&mw, w.W2, rows, kD, 64, 64, true) ||
        !make_map(&mq, w.Q2, rows, kD, 64, 64, true) ||
        !make_map(&mk, w.Kb2, rows, kD, 64, 64, true) ||
        !make_map(&ma, w.Aqk2, (uint64_t)BH * NT * kC, kC, 64, 64, true) ||
        !make_map(&mu, w.U2, rows, kD, 128, 64, false))
        return KDA_ERR_CUDA;
    // chunk-start states, [BH*NT*V][K]: 64-column boxes of 128 rows (a dummy
    // map over W when no states are kept)
    // and delta, [BH*NT*V][C]: one box of 128 rows
    if ((h_out == nullptr) != (delta_out == nullptr)) return KDA_ERR_INVALID_ARG;
    if ((u_lo == nullptr) != (delta_lo == nullptr) || (delta_lo && (!delta_out || nseg >= 3)) ||
        (vl && nseg >= 3))
        return KDA_ERR_INVALID_ARG;
    CUtensorMap mh, mdl, mo;
    if (!(h_out ? make_map(&mh, h_out, (uint64_t)BH * NT * kD, kD, 64, 128, true)
                : make_map(&mh, w.W2, rows, kD, 64, 64, true)) ||
        !(delta_out ? make_map(&mdl, delta_out, (uint64_t)BH * NT * kD, kC, 64, 128, true)
                    : make_map(&mdl, w.W2, rows, kD, 64, 64, true)))
        return KDA_ERR_CUDA;
    // the output o [B*T][HV][V] in [64 t][64 v] boxes (a dummy map over W when
    // there is no output)
    if (!(o ? make_map_tok(&mo, o, tok_rows(d, vl), d.HV, d.V) : make_map_tok(&mo, w.W2, rows, 1, kD)))
        return KDA_ERR_CUDA;
    ChainArgs args;
    args.B = d.B;
    args.T = d.T;
    args.HV = d.HV;
    args.NT = NT;
    args.D = d.K;
    args.gam = gam;
    args.h0 = h0;
    args.o = static_cast<__nv_bfloat16*>(o);
    args.ht = ht;
    args.h_out = h_out;
    args.delta_out = delta_out;
    args.u_lo = u_lo;
    args.delta_lo = delta_lo;
    args.nseg = 0;
    args.seglen = 0;
    args.pass = 0;
    args.sbuf = args.zbuf = args.mbuf = nullptr;
    args.ident = nullptr;
    args.ctab = vl ? vl->ctab : nullptr;
    args.sfirst = vl ? vl->sfirst : nullptr;
    auto chain = vl ? (delta_lo ? chain_fwd_kernel<true, true> : chain_fwd_kernel<false, true>)
                    : (delta_lo ? chain_fwd_kernel<true, false> : chain_fwd_kernel<false, false>);
    if (cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)CHAIN_SMEM) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (nseg < 3) {
        // three roles, timed apart: forward (o), saving forward (o and the
        // chunk-start states), and the backward's recompute (states only)
        TimedLaunch tl(!h_out ? "tc_chain_fwd" : o ? "tc_chain_fwd_save" : "tc_chain_states", s);
        chain<<<ctas, kChainThreads, CHAIN_SMEM, s>>>(mw, mq, mk, ma, mu, mh, mdl, mo, args);
        return launch_status();
    }
    // segmented: pass 1 (segment 0 in full; later segments from zero and as
    // transitions), the combine step, pass 3 (later segments in full)
    args.nseg = nseg;
    args.seglen = (NT + nseg - 1) / nseg;
    args.sbuf = w.sbuf;
    args.zbuf = w.zbuf;
    args.mbuf = w.mbuf;
    args.ident = w.ident;
    const int D = d.K;
    const size_t cbytes = ((size_t)D * (D + 4) + (size_t)D * D) * sizeof(float);
    if (cudaFuncSetAttribute(chain_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)cbytes) != cudaSuccess)
        return KDA_ERR_CUDA;
    fill_identity_kernel<<<(D * D + 255) / 256, 256, 0, s>>>(w.ident, D);
    kda_status st;
    if ((st = launch_status()) != KDA_OK) return st;
    {
        TimedLaunch tl("tc_chain_seg_pass1", s);
        args.pass = 1;
        chain<<<BH * (2 * nseg - 3), kChainThreads, CHAIN_SMEM, s>>>(
            mw, mq, mk, ma, mu, mh, mdl, mo, args);
    }
    if ((st = launch_status()) != KDA_OK) return st;
    {
        TimedLaunch tl("tc_chain_seg_combine", s);
        chain_combine_kernel<<<BH, 256, cbytes, s>>>(D, nseg, w.sbuf, w.zbuf, w.mbuf);
    }
    if ((st = launch_status()) != KDA_OK) return st;
    {
        TimedLaunch tl("tc_chain_seg_pass3", s);
        args.pass = 3;
        chain<<<BH * (nseg - 1), kChainThreads, CHAIN_SMEM, s>>>(
            mw, mq, mk, ma, mu, mh, mdl, mo, args);
    }
    return launch_status();
}

}  // namespace

// K = V = 128, or K = V = 64 run at 128 with the upper channels zero (the
// tensor maps fill them on load and skip them on store; the plain global
// accesses of states and gradients use the tensors' own width).
bool tc_supported(const kda_dims& d) {
    return d.dtype == KDA_BF16 && d.K == d.V && (d.K == kD || d.K == 64) && d.chunk_size == kC &&
           get_encoder() != nullptr;
}

size_t tc_workspace_bytes(const kda_dims& d, int for_bwd) {
    return tc_carve(d, for_bwd ? 1 : 0, nullptr, nullptr);
}

kda_status tc_fwd(const kda_dims& d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, void* o, float* ht, void* ws, bool save,
                  cudaStream_t s) {
    TcWs w;
    tc_carve(d, save ? 1 : 0, static_cast<char*>(ws), &w);
    float* gam = nullptr;
    kda_status st = run_intra_tc(d, w, q, k, v, g, beta, save, s, &gam);
    if (st != KDA_OK) return st;
    if (save) return run_chain_fwd(d, w, gam, h0, o, ht, w.h2, w.d2, s);
    // the plain forward cuts long sequences into segments when few heads
    // would leave most SMs idle during the state pass
    return run_chain_fwd(d, w, gam, h0, o, ht, nullptr, nullptr, s, chain_segments(d));
}

namespace {
// The backward on a carved workspace; vl: a packed batch (d then has B = 1
// and the padded T), or null.
kda_status tc_bwd_run(const kda_dims& d, const TcWs& w, const TcVl* vl, const void* q,
                      const void* k, const void* v, const void* g, const void* beta,
                      const float* h0, const void* dout, const float* dht, void* dq, void* dk,
                      void* dv, void* dg, void* dbeta, float* dh0, bool from_saved,
                      cudaStream_t s) {
    float* gam = nullptr;
    kda_status st = KDA_OK;
    // An upstream final-state gradient runs the two-term path: U, Kb, delta
    // and dS also leave their kernels as bf16 low parts, and the contractions
    // over V take grad_v_px_kernel.  The saving forward keeps no low parts,
    // so this path always recomputes.
    const bool px = dht != nullptr;
    const int BH = d.B * d.HV, NT = d.T / kC;
    const uint64_t rows = (uint64_t)BH * d.T;
    // reverse chain, on stream rs: dS and ddelta from dO and the intra-chunk
    // quantities alone (the forward states do not enter)
    auto run_chain_rev = [&](cudaStream_t rs) -> kda_status {
        CUtensorMap mdo, mq, mw, mk, ma, mdh, mddst;
        if (!make_map(&mdh, w.dh2, (uint64_t)BH * NT * kD, kD, 64, 128, true) ||
            !make_map_tok(&mdo, dout, tok_rows(d, vl), d.HV, d.V) ||
            !make_map(&mq, w.Q2, rows, kD, 64, 64, true) ||
            !make_map(&mw, w.W2, rows, kD, 64, 64, true) ||
            !make_map(&mk, w.Kb2, rows, kD, 64, 64, true) ||
            !make_map(&ma, w.Aqk2, (uint64_t)BH * NT * kC, kC, 64, 64, true) ||
            !make_map(&mddst, w.dd2, rows, kD, 64, 64, true))   // ddelta [BH*T][V]
            return KDA_ERR_CUDA;
        ChainBwdArgs a;
        a.B = d.B;
        a.T = d.T;
        a.HV = d.HV;
        a.NT = NT;
        a.D = d.K;
        a.gam = gam;
        a.dht = dht;
        a.dh0 = dh0;
        a.dh_out = w.dh2;
        a.dh_lo = px ? w.dhlo : nullptr;
        a.ctab = vl ? vl->ctab : nullptr;
        a.sfirst = vl ? vl->sfirst : nullptr;
        auto kern = vl ? (px ? chain_bwd_kernel<true, true> : chain_bwd_kernel<false, true>)
                       : (px ? chain_bwd_kernel<true, false> : chain_bwd_kernel<false, false>);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)CHAIN_SMEM) != cudaSuccess)
            return KDA_ERR_CUDA;
        TimedLaunch tl("tc_chain_bwd", rs);
        kern<<<vl ? vl->nseq * d.HV : BH, kChainThreads, CHAIN_SMEM, rs>>>(mdo, mq, mw, mk, ma,
                                                                          mdh, mddst, a);
        return launch_status();
    };
    if (from_saved && !px) {
        SimtWsPtrs p0;
        simt_ws_ptrs(tc_wide(d), 0, w.simt, &p0);  // where the intra kernel left gam
        gam = p0.gam;
        if ((st = run_chain_rev(s)) != KDA_OK) return st;
    } else {
        if ((st = run_intra_tc(d, w, q, k, v, g, beta, true, s, &gam, px ? w.Ulo : nullptr,
                               px ? w.Kblo : nullptr, vl)) != KDA_OK)
            return st;
        // forward recompute (chunk-start states and delta) and the reverse
        // pass.  Without an upstream final-state gradient the two read only
        // the intra-chunk quantities and write disjoint arrays, and each
        // fills one SM per (sequence, head): they run side by side, the
        // reverse pass on a second stream.  With one, the reverse pass writes
        // dS's low parts over U's, which the forward pass reads first.
        cudaStream_t as = px ? nullptr : aux_stream();
        if (!as) {
            if ((st = run_chain_fwd(d, w, gam, h0, nullptr, nullptr, w.h2, w.d2, s, 0,
                                    px ? w.Ulo : nullptr, px ? w.d2lo : nullptr, vl)) != KDA_OK)
                return st;
            if ((st = run_chain_rev(s)) != KDA_OK) return st;
        } else {
            cudaEvent_t fork = nullptr, join = nullptr;
            if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
                if (fork) cudaEventDestroy(fork);
                return KDA_ERR_CUDA;
            }
            kda_status st_rev = KDA_ERR_CUDA;
            if (cudaEventRecord(fork, s) == cudaSuccess &&
                cudaStreamWaitEvent(as, fork, 0) == cudaSuccess) {
                st_rev = run_chain_rev(as);
                st = run_chain_fwd(d, w, gam, h0, nullptr, nullptr, w.h2, w.d2, s, 0, nullptr,
                                   nullptr, vl);
                // the join is recorded whatever the launches returned, so
                // that the caller's stream always waits for the second one
                if (cudaEventRecord(join, as) != cudaSuccess ||
                    cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
                    st_rev = KDA_ERR_CUDA;
            }
            cudaEventDestroy(fork);
            cudaEventDestroy(join);
            if (st_rev != KDA_OK) return st_rev;
            if (st != KDA_OK) return st;
        }
    }
    // contractions over V
    {
        SimtWsPtrs p;
        simt_ws_ptrs(tc_wide(d), 1, w.simt, &p);
        CUtensorMap mh, mdh, mdo, mdd, md, mv, mt;
        const uint64_t srows = (uint64_t)BH * NT * kD;
        if (!make_map(&mh, w.h2, srows, kD, 64, 128, true) ||
            !make_map(&mdh, w.dh2, srows, kD, 64, 128, true) ||
            !make_map_tok(&mdo, dout, tok_rows(d, vl), d.HV, d.V) ||
            !make_map(&mdd, w.dd2, rows, kD, 64, 64, true) ||
            !make_map(&md, w.d2, srows, kC, 64, 128, true) ||
            !make_map_tok(&mv, v, tok_rows(d, vl), d.HV, d.V) ||
            !make_map(&mt, w.T2, (uint64_t)BH * NT * kC, kC, 64, 64, true))
            return KDA_ERR_CUDA;
        GradArgs a;
        a.T = d.T;
        a.HV = d.HV;
        a.NT = NT;
        a.D = d.V;
        a.BH = BH;
        a.beta = static_cast<const __nv_bfloat16*>(beta);
        a.dv = static_cast<__nv_bfloat16*>(dv);
        a.dQh = p.dQh;
        a.dW = reinterpret_cast<__nv_bfloat16*>(p.dWm);  // bf16 in the fp32 array's space
        a.dKb = p.dKb;
        a.dgam = p.dgam;
        a.dAqk = reinterpret_cast<__nv_bfloat16*>(p.dAqk);
        a.dTv = p.dTv;
        a.dbv = p.dbv;
        a.ctab = vl ? vl->ctab : nullptr;
        if (px) {
            CUtensorMap mdhl, mdl, mkb, mkbl, ma;
            if (!make_map(&mdhl, w.dhlo, srows, kD, 64, 128, true) ||
                !make_map(&mdl, w.d2lo, srows, kC, 64, 128, true) ||
                !make_map(&mkb, w.Kb2, rows, kD, 64, 64, true) ||
                !make_map(&mkbl, w.Kblo, rows, kD, 64, 64, true) ||
                !make_map(&ma, w.Aqk2, (uint64_t)BH * NT * kC, kC, 64, 64, true))
                return KDA_ERR_CUDA;
            auto kern = d.V == kD ? (vl ? grad_v_px_kernel<kD, true> : grad_v_px_kernel<kD, false>)
                                  : (vl ? grad_v_px_kernel<64, true> : grad_v_px_kernel<64, false>);
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)PX_SMEM) != cudaSuccess)
                return KDA_ERR_CUDA;
            TimedLaunch tl("tc_grad_v_px", s);
            kern<<<std::min(BH * NT, sm_count()), kGradThreads, PX_SMEM, s>>>(
                mh, mdh, mdhl, mdo, md, mdl, mkb, mkbl, ma, mv, mt, a);
        } else {
            CUtensorMap mdqh, mdkb;   // the fp32 outputs [BH*T][128], one box per chunk
            if (!make_map_f32(&mdqh, p.dQh, rows, kD, kD, kC) ||
                !make_map_f32(&mdkb, p.dKb, rows, kD, kD, kC))
                return KDA_ERR_CUDA;
            auto kern = d.V == kD ? (vl ? grad_v_kernel<kD, true> : grad_v_kernel<kD, false>)
                                  : (vl ? grad_v_kernel<64, true> : grad_v_kernel<64, false>);
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)GRAD_SMEM) != cudaSuccess)
                return KDA_ERR_CUDA;
            TimedLaunch tl("tc_grad_v", s);
            // persistent: one CTA per SM walks the chunks
            kern<<<std::min(BH * NT, sm_count()), kGradThreads, GRAD_SMEM, s>>>(
                mh, mdh, mdo, mdd, md, mv, mt, mdqh, mdkb, a);
        }
    }
    if ((st = launch_status()) != KDA_OK) return st;
    SimtWsPtrs p;
    simt_ws_ptrs(tc_wide(d), 1, w.simt, &p);
    if ((st = run_local_bwd_tc(d, w, p, q, k, g, beta, dq, dk, dg, dbeta, s, vl)) != KDA_OK)
        return st;
    if (d.HV == d.H && !d.qk_l2norm) return KDA_OK;
    kda_dims dt = d;   // the token rows of the dq, dk arrays
    if (vl) dt.T = vl->Ttok;
    return group_sum_launch(dt, p.dqh, p.dkh, q, k, dq, dk, s);
}

// Padded dims of a packed batch (the SIMT kernels use the same bound): B = 1
// and ceil(T / 64) + nseq chunk slots.
kda_dims tc_varlen_dims(const kda_dims& d, int nseq) {
    kda_dims p = d;
    p.B = 1;
    p.T = ((d.T + kC - 1) / kC + nseq) * kC;
    return p;
}
// The workspace of a packed batch: the tensor-core carve of the padded dims,
// then the chunk table [NT][2] and the first chunk slot of every sequence.
size_t tc_varlen_carve(const kda_dims& d, int nseq, int for_bwd, char* base, TcWs* w,
                       TcVl* vl) {
    const kda_dims p = tc_varlen_dims(d, nseq);
    size_t off = tc_carve(p, for_bwd, base, w);
    int* ctab = base ? reinterpret_cast<int*>(base + off) : nullptr;
    off += align256((size_t)(p.T / kC) * 2 * sizeof(int));
    int* sfirst = base ? reinterpret_cast<int*>(base + off) : nullptr;
    off += align256((size_t)(nseq + 1) * sizeof(int));
    if (vl) *vl = TcVl{ctab, sfirst, nseq, d.T};
    return off;
}
}  // namespace

kda_status tc_bwd(const kda_dims& d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, const void* dout, const float* dht,
                  void* dq, void* dk, void* dv, void* dg, void* dbeta, float* dh0, void* ws,
                  bool from_saved, cudaStream_t s) {
    TcWs w;
    tc_carve(d, 1, static_cast<char*>(ws), &w);
    return tc_bwd_run(d, w, nullptr, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0,
                      from_saved, s);
}

size_t tc_varlen_workspace_bytes(const kda_dims& d, int nseq, int for_bwd) {
    return tc_varlen_carve(d, nseq, for_bwd ? 1 : 0, nullptr, nullptr, nullptr);
}

kda_status tc_fwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0, void* o,
                         float* ht, void* ws, bool save, cudaStream_t s) {
    TcWs w;
    TcVl vl;
    tc_varlen_carve(d, nseq, save ? 1 : 0, static_cast<char*>(ws), &w, &vl);
    const kda_dims p = tc_varlen_dims(d, nseq);
    kda_status st = varlen_table_launch(cu, nseq, d.T, kC, p.T / kC, const_cast<int*>(vl.ctab),
                                        const_cast<int*>(vl.sfirst), s);
    if (st != KDA_OK) return st;
    float* gam = nullptr;
    if ((st = run_intra_tc(p, w, q, k, v, g, beta, save, s, &gam, nullptr, nullptr, &vl)) != KDA_OK)
        return st;
    return run_chain_fwd(p, w, gam, h0, o, ht, save ? w.h2 : nullptr, save ? w.d2 : nullptr, s, 0,
                         nullptr, nullptr, &vl);
}

kda_status tc_bwd_varlen(const kda_dims& d, const int* cu, int nseq, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0,
                         const void* dout, const float* dht, void* dq, void* dk, void* dv,
                         void* dg, void* dbeta, float* dh0, void* ws, bool from_saved,
                         cudaStream_t s) {
    TcWs w;
    TcVl vl;
    tc_varlen_carve(d, nseq, 1, static_cast<char*>(ws), &w, &vl);
    const kda_dims p = tc_varlen_dims(d, nseq);
    kda_status st = varlen_table_launch(cu, nseq, d.T, kC, p.T / kC, const_cast<int*>(vl.ctab),
                                        const_cast<int*>(vl.sfirst), s);
    if (st != KDA_OK) return st;
    // (the table is rebuilt from cu_seqlens even after a saving forward)
    return tc_bwd_run(p, w, &vl, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0,
                      from_saved, s);
}

namespace {
// Diagnostic of the bounded-wait error path: one warp waits, with a limit of
// `limit` cycles, on an mbarrier that nothing arrives at.  The wait gives up,
// records its code in the error word and the kernel returns; nothing is in
// flight, so the context stays usable.
__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    wait_bar_limit(&bar, 0, 99, limit);
}
}  // namespace

kda_status tc_selftest_timeout(long long limit_cycles, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(limit_cycles);
    return launch_status();
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
