// Tensor-core (tcgen05 + TMEM + TMA) chunk scan for bf16, K = V = 128,
// chunk 64.
//
// Forward state pass ("chain") of the chunk form (K3 README, table 实现路线表,
// row L2, step (4): the state passed between chunks).  One CTA per (b, hv)
// walks the chunks in order and keeps the K x V state S on chip, as fp32 in
// tensor memory.  Everything is computed transposed so that the MMA M
// dimension is the value dimension (128 rows = 128 TMEM lanes):
//     D12W  = S^T W^T            (M=128 v, N=64 rows, K=128 k)
//     delta^T = U^T - D12W       (epilogue, fp32 -> bf16 operand in smem)
//     O^T   = S^T Qh^T + delta^T Aqk^T
//     S^T   = diag(gam) S^T + delta^T Kb       (gam applied by the epilogue)
// Per-chunk operands (W, Qh, Kb^T, Aqk, U as bf16; gam fp32) arrive by TMA
// into a two-stage ring.  Warp roles: warp 0 issues TMA, warp 1 owns TMEM and
// issues MMAs (one thread), warps 2-5 are the epilogue (one TMEM lane per
// value column).  Every mbarrier wait is bounded: on expiry the kernel records
// an error code in g_tc_error and unwinds.
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
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 255u) == 0) {
            if (*reinterpret_cast<volatile int*>(&g_tc_error) != 0) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                atomicCAS(&g_tc_error, 0, code);
                return false;
            }
        }
    }
    return true;
}
// Warp-uniform version: every lane waits, the warp proceeds only if all did.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, int code) {
    const bool ok = wait_bar(bar, parity, code);
    return __all_sync(0xffffffffu, ok);
}

// ---- shared-memory plan of the chain kernel (offsets from a 1024-aligned base) ----
constexpr uint32_t OFF_W = 0;          // 64 rows x 128 bf16, 2 k-blocks of 8 KB
constexpr uint32_t OFF_Q = 16384;      // same for Qh
constexpr uint32_t OFF_KBT = 32768;    // Kb^T: 128 rows (k) x 64 bf16 (c)
constexpr uint32_t OFF_AQK = 49152;    // Aqk: 64 rows x 64 bf16
constexpr uint32_t OFF_U = 57344;      // U: 64 x 128 bf16, row-major, unswizzled
constexpr uint32_t OFF_GAM = 73728;    // gam: 128 fp32
constexpr uint32_t STAGE_BYTES = 74752;
constexpr uint32_t STAGE_TX = 16384 * 2 + 16384 + 8192 + 16384 + 512;
constexpr uint32_t OFF_S = 2 * STAGE_BYTES;    // S^T operand: 128 rows x 128 bf16 (2 k-blocks)
constexpr uint32_t OFF_DELTA = OFF_S + 32768;  // delta^T operand: 128 rows x 64 bf16
constexpr uint32_t OFF_BAR = OFF_DELTA + 16384;
constexpr uint32_t CHAIN_SMEM = OFF_BAR + 256 + 1024;  // + alignment slack

// TMEM columns
constexpr uint32_t TM_S = 0, TM_W = 128, TM_O0 = 192, TM_O1 = 256, TM_COLS = 512;

struct ChainArgs {
    int B, T, HV, NT;
    const float* gam;   // [BH*NT][128]
    const float* h0;    // [BH][K][V] or null
    __nv_bfloat16* o;   // [B,T,HV,V]
    float* ht;          // [BH][K][V] or null
    float* h_out;       // [BH][NT][K][V] or null (states at chunk starts)
    __nv_bfloat16* delta_out;  // [BH*T][V] or null
};

__global__ void __launch_bounds__(192, 1)
chain_fwd_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_kbt,
                 const __grid_constant__ CUtensorMap tm_aqk,
                 const __grid_constant__ CUtensorMap tm_u, ChainArgs a) {
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
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(full + 9);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / a.HV, hv = bh % a.HV;
    const int NT = a.NT;

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&empty[0], 129);
        mbar_init(&empty[1], 129);
        mbar_init(bar_S, 128);
        mbar_init(bar_delta, 128);
        mbar_init(bar_D12, 1);
        mbar_init(bar_D3, 1);
        mbar_init(bar_fin, 1);
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
            int issued = 0;
            for (int n = 0; n < NT; ++n) {
                const int s = n & 1;
                if (!wait_bar(&empty[s], ((n >> 1) & 1) ^ 1, 1)) break;
                uint8_t* st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], STAGE_TX);
                const int row = bh * a.T + n * kC;
                const int crow = bh * NT + n;
                tma_load_2d(st + OFF_W, &tm_w, &full[s], 0, row);
                tma_load_2d(st + OFF_W + 8192, &tm_w, &full[s], 64, row);
                tma_load_2d(st + OFF_Q, &tm_q, &full[s], 0, row);
                tma_load_2d(st + OFF_Q + 8192, &tm_q, &full[s], 64, row);
                tma_load_2d(st + OFF_KBT, &tm_kbt, &full[s], 0, crow * kD);
                tma_load_2d(st + OFF_AQK, &tm_aqk, &full[s], 0, crow * kC);
                tma_load_2d(st + OFF_U, &tm_u, &full[s], 0, row);
                bulk_load(st + OFF_GAM, a.gam + (size_t)crow * kD, 512, &full[s]);
                issued = n + 1;
            }
            // do not leave copies in flight: wait for the last stages issued
            for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n)
                wait_bar(&full[n & 1], (n >> 1) & 1, 2);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc64 = idesc_bf16_f32(128, 64);
            const uint32_t idesc128 = idesc_bf16_f32(128, 128);
            const uint32_t sS = smem_u32(smem + OFF_S), sD = smem_u32(smem + OFF_DELTA);
            for (int n = 0; n < NT; ++n) {
                const int s = n & 1;
                const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
                if (!wait_bar(&full[s], (n >> 1) & 1, 3)) break;
                if (!wait_bar(bar_S, n & 1, 4)) break;
                tc_fence_after();
                const uint32_t tO = tmem + ((n & 1) ? TM_O1 : TM_O0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t kb = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_W, sdesc_sw128(sS + ka), sdesc_sw128(st + OFF_W + kb),
                             idesc64, kk > 0);
                }
                mma_commit(bar_D12);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t kb = (kk >> 2) * 8192 + (kk & 3) * 32;
                    mma_bf16(tO, sdesc_sw128(sS + ka), sdesc_sw128(st + OFF_Q + kb), idesc64,
                             kk > 0);
                }
                if (!wait_bar(bar_delta, n & 1, 5)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_S, sdesc_sw128(sD + kk * 32),
                             sdesc_sw128(st + OFF_KBT + kk * 32), idesc128, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tO, sdesc_sw128(sD + kk * 32), sdesc_sw128(st + OFF_AQK + kk * 32),
                             idesc64, 1);
                mma_commit(bar_D3);
                mma_commit(&empty[s]);
            }
            // all issued MMAs complete before TMEM is released
            mma_commit(bar_fin);
            wait_bar(bar_fin, 0, 6);
        }
    } else {
        // ---------------- epilogue: thread <-> value column v ----------------
        const int q = warp & 3;
        const int v = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint8_t* sS = smem + OFF_S;
        uint8_t* sDelta = smem + OFF_DELTA;
        float r[32];
        bool ok = true;

        // E1: bring S_n to the bf16 operand tile, scale the TMEM copy by gam_n.
        auto e1 = [&](int n) -> bool {
            const int s = n & 1;
            if (!wait_bar_warp(&full[s], (n >> 1) & 1, 7)) return false;
            const float* gam = reinterpret_cast<const float*>(smem + s * STAGE_BYTES + OFF_GAM);
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                if (n == 0) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = a.h0 ? a.h0[((size_t)bh * kD + cb * 32 + i) * kD + v] : 0.f;
                } else {
                    tmem_ld32(tmem + lane_off + TM_S + cb * 32, r);
                }
                if (a.h_out) {
                    float* hp = a.h_out + (((size_t)bh * NT + n) * kD + cb * 32) * kD + v;
#pragma unroll
                    for (int i = 0; i < 32; ++i) hp[(size_t)i * kD] = r[i];
                }
                uint8_t* base = sS + (cb >> 1) * 16384;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 pk;
                    pk.x = pack_bf16(r[8 * j + 0], r[8 * j + 1]);
                    pk.y = pack_bf16(r[8 * j + 2], r[8 * j + 3]);
                    pk.z = pack_bf16(r[8 * j + 4], r[8 * j + 5]);
                    pk.w = pack_bf16(r[8 * j + 6], r[8 * j + 7]);
                    *reinterpret_cast<uint4*>(base + sw128_offset(v, (cb & 1) * 32 + 8 * j)) = pk;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] *= gam[cb * 32 + i];
                tmem_st32(tmem + lane_off + TM_S + cb * 32, r);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_S);
            return true;
        };

        ok = e1(0);
        for (int n = 0; ok && n < NT; ++n) {
            const int s = n & 1;
            // E2: delta^T = U^T - S^T W^T  -> bf16 operand tile
            if (!wait_bar_warp(bar_D12, n & 1, 8)) { ok = false; break; }
            tc_fence_after();
            const __nv_bfloat16* U =
                reinterpret_cast<const __nv_bfloat16*>(smem + s * STAGE_BYTES + OFF_U);
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                tmem_ld32(tmem + lane_off + TM_W + cb * 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    r[i] = __bfloat162float(U[(cb * 32 + i) * kD + v]) - r[i];
                if (a.delta_out) {
                    __nv_bfloat16* dp =
                        a.delta_out + ((size_t)bh * a.T + (size_t)n * kC + cb * 32) * kD + v;
#pragma unroll
                    for (int i = 0; i < 32; ++i) dp[(size_t)i * kD] = __float2bfloat16_rn(r[i]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 pk;
                    pk.x = pack_bf16(r[8 * j + 0], r[8 * j + 1]);
                    pk.y = pack_bf16(r[8 * j + 2], r[8 * j + 3]);
                    pk.z = pack_bf16(r[8 * j + 4], r[8 * j + 5]);
                    pk.w = pack_bf16(r[8 * j + 6], r[8 * j + 7]);
                    *reinterpret_cast<uint4*>(sDelta + sw128_offset(v, cb * 32 + 8 * j)) = pk;
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_delta);
            mbar_arrive(&empty[s]);

            if (!wait_bar_warp(bar_D3, n & 1, 9)) { ok = false; break; }
            tc_fence_after();
            if (n + 1 < NT) {
                if (!e1(n + 1)) { ok = false; break; }
            } else if (a.ht) {
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    tmem_ld32(tmem + lane_off + TM_S + cb * 32, r);
                    float* hp = a.ht + ((size_t)bh * kD + cb * 32) * kD + v;
#pragma unroll
                    for (int i = 0; i < 32; ++i) hp[(size_t)i * kD] = r[i];
                }
            }
            // E3: output rows of chunk n
            const uint32_t tO = (n & 1) ? TM_O1 : TM_O0;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                tmem_ld32(tmem + lane_off + tO + cb * 32, r);
                __nv_bfloat16* op =
                    a.o + (((size_t)b * a.T + (size_t)n * kC + cb * 32) * a.HV + hv) * kD + v;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    op[(size_t)i * a.HV * kD] = __float2bfloat16_rn(r[i]);
            }
        }
        (void)ok;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// Converts the fp32 per-chunk quantities of the SIMT intra kernel into the
// bf16 operand layouts of the chain kernel.
__global__ void pack_operands_kernel(int BH, int T, int NT, const float* __restrict__ W,
                                     const float* __restrict__ Qh, const float* __restrict__ U,
                                     const float* __restrict__ Kb, const float* __restrict__ Aqk,
                                     __nv_bfloat16* __restrict__ W2, __nv_bfloat16* __restrict__ Q2,
                                     __nv_bfloat16* __restrict__ U2,
                                     __nv_bfloat16* __restrict__ KbT2,
                                     __nv_bfloat16* __restrict__ Aqk2) {
    const size_t nrow = (size_t)BH * T * kD;
    const size_t ncc = (size_t)BH * NT * kC * kC;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nrow;
         i += (size_t)gridDim.x * blockDim.x) {
        W2[i] = __float2bfloat16_rn(W[i]);
        Q2[i] = __float2bfloat16_rn(Qh[i]);
        U2[i] = __float2bfloat16_rn(U[i]);
        // KbT2[(chunk*128 + k)*64 + c] = Kb[(chunk*64 + c)*128 + k]
        const size_t chunk = i / (kC * kD), rem = i % (kC * kD);
        const size_t k = rem / kC, c = rem % kC;
        KbT2[i] = __float2bfloat16_rn(Kb[(chunk * kC + c) * kD + k]);
        if (i < ncc) Aqk2[i] = __float2bfloat16_rn(Aqk[i]);
    }
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

struct TcWs {
    char* simt;                      // SIMT intra workspace (fp32 quantities)
    __nv_bfloat16 *W2, *Q2, *U2, *KbT2, *Aqk2;
};

size_t tc_carve(const kda_dims& d, char* base, TcWs* w) {
    const size_t BH = (size_t)d.B * d.HV, T = d.T, NT = d.T / kC;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    TcWs x{};
    x.simt = take(simt_workspace_bytes(d, 0));
    x.W2 = reinterpret_cast<__nv_bfloat16*>(take(BH * T * kD * 2));
    x.Q2 = reinterpret_cast<__nv_bfloat16*>(take(BH * T * kD * 2));
    x.U2 = reinterpret_cast<__nv_bfloat16*>(take(BH * T * kD * 2));
    x.KbT2 = reinterpret_cast<__nv_bfloat16*>(take(BH * NT * kD * kC * 2));
    x.Aqk2 = reinterpret_cast<__nv_bfloat16*>(take(BH * NT * kC * kC * 2));
    if (w) *w = x;
    return off;
}

}  // namespace

bool tc_supported(const kda_dims& d) {
    return d.dtype == KDA_BF16 && d.K == kD && d.V == kD && d.chunk_size == kC &&
           get_encoder() != nullptr;
}

size_t tc_workspace_bytes(const kda_dims& d, int for_bwd) {
    if (for_bwd) return simt_workspace_bytes(d, 1);
    return tc_carve(d, nullptr, nullptr);
}

kda_status tc_fwd(const kda_dims& d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, void* o, float* ht, void* ws,
                  cudaStream_t s) {
    TcWs w;
    tc_carve(d, static_cast<char*>(ws), &w);
    SimtIntraOut io;
    kda_status st = simt_intra_only(d, q, k, v, g, beta, w.simt, &io, s);
    if (st != KDA_OK) return st;
    const int BH = d.B * d.HV, NT = d.T / kC;
    {
        TimedLaunch tl("tc_pack", s);
        pack_operands_kernel<<<152 * 8, 256, 0, s>>>(BH, d.T, NT, io.W, io.Qh, io.U, io.Kb, io.Aqk,
                                                     w.W2, w.Q2, w.U2, w.KbT2, w.Aqk2);
    }
    if ((st = launch_status()) != KDA_OK) return st;
    CUtensorMap mw, mq, mk, ma, mu;
    const uint64_t rows = (uint64_t)BH * d.T;
    if (!make_map(&mw, w.W2, rows, kD, 64, 64, true) ||
        !make_map(&mq, w.Q2, rows, kD, 64, 64, true) ||
        !make_map(&mk, w.KbT2, (uint64_t)BH * NT * kD, kC, 64, 128, true) ||
        !make_map(&ma, w.Aqk2, (uint64_t)BH * NT * kC, kC, 64, 64, true) ||
        !make_map(&mu, w.U2, rows, kD, 128, 64, false))
        return KDA_ERR_CUDA;
    ChainArgs args;
    args.B = d.B;
    args.T = d.T;
    args.HV = d.HV;
    args.NT = NT;
    args.gam = io.gam;
    args.h0 = h0;
    args.o = static_cast<__nv_bfloat16*>(o);
    args.ht = ht;
    args.h_out = nullptr;
    args.delta_out = nullptr;
    if (cudaFuncSetAttribute(chain_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)CHAIN_SMEM) != cudaSuccess)
        return KDA_ERR_CUDA;
    {
        TimedLaunch tl("tc_chain_fwd", s);
        chain_fwd_kernel<<<BH, 192, CHAIN_SMEM, s>>>(mw, mq, mk, ma, mu, args);
    }
    return launch_status();
}

kda_status tc_bwd(const kda_dims& d, const void* q, const void* k, const void* v, const void* g,
                  const void* beta, const float* h0, const void* dout, const float* dht,
                  void* dq, void* dk, void* dv, void* dg, void* dbeta, float* dh0, void* ws,
                  cudaStream_t s) {
    // The backward runs the SIMT kernels until its tensor-core kernels land.
    return simt_bwd(d, q, k, v, g, beta, h0, dout, dht, dq, dk, dv, dg, dbeta, dh0, ws, s);
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
