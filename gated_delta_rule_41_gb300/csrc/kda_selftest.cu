// Self-test of the tensor-core building blocks used by the chunk kernels:
// one D[128 x N] = A[128 x 64] * B[N x 64]^T product with bf16 operands in
// 128B-swizzled K-major shared-memory tiles, an fp32 accumulator in TMEM, and
// the result read back with tcgen05.ld.  Operands are staged either by TMA or
// by threads writing the swizzled layout directly (the two ways the chunk
// kernels fill operand tiles).
#include "kda_common.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows) {
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return reinterpret_cast<EncodeFn>(p)(
               m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 128 threads.  smem (160 KB, so that any stride reading stays in bounds):
// A tile at 0 (16 KB), B tile at 64 KB (up to 16 KB), barriers at 144 KB.
// flags: bit0 TMA staging, bit1 A MN-major, bit2 B MN-major.  MN-major
// operands use the chunk kernels' descriptor (64-element M/N blocks 8 KB
// apart, 8-row K groups 1 KB apart).
__global__ void __launch_bounds__(128, 1)
selftest_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                float* __restrict__ D, int N, int flags, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int use_tma = flags & 1, a_mn = (flags >> 1) & 1, b_mn = (flags >> 2) & 1;
    uint8_t* sA = smem;
    uint8_t* sB = smem + 65536;
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + 147456);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar_tma + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(holder, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;

    if (use_tma) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(bar_tma, (128 + N) * 128);
            // K-major: one box of 64 (k) x rows.  MN-major: boxes of 64 (m/n) x 64 (k),
            // consecutive 64-element M/N blocks 8 KB apart.
            if (a_mn) {
                tma_load_2d(sA, &ma, bar_tma, 0, 0);
                tma_load_2d(sA + 8192, &ma, bar_tma, 64, 0);
            } else {
                tma_load_2d(sA, &ma, bar_tma, 0, 0);
            }
            if (b_mn) {
                for (int nb = 0; nb < N / 64; ++nb)
                    tma_load_2d(sB + nb * 8192, &mb, bar_tma, nb * 64, 0);
            } else {
                tma_load_2d(sB, &mb, bar_tma, 0, 0);
            }
        }
    } else {
        for (int i = threadIdx.x; i < 128 * 8; i += 128) {
            const int r = i / 8, c8 = i % 8;
            *reinterpret_cast<uint4*>(sA + sw128_offset(r, c8 * 8)) =
                *reinterpret_cast<const uint4*>(A + r * 64 + c8 * 8);
        }
        for (int i = threadIdx.x; i < N * 8; i += 128) {
            const int r = i / 8, c8 = i % 8;
            *reinterpret_cast<uint4*>(sB + sw128_offset(r, c8 * 8)) =
                *reinterpret_cast<const uint4*>(B + r * 64 + c8 * 8);
        }
        fence_async_smem();
    }
    __syncthreads();
    bool ok = true;
    if (use_tma) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar_tma, 0))
            if (clock64() - t0 > 2000000000LL) { ok = false; break; }
    }
    if (threadIdx.x == 0 && ok) {
        tc_fence_after();
        const uint32_t idesc =
            idesc_bf16_f32(128, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = a_mn ? sdesc_mn_sw128(smem_u32(sA) + kk * 2048, 8192)
                                     : sdesc_sw128(smem_u32(sA) + kk * 32);
            const uint64_t bd = b_mn ? sdesc_mn_sw128(smem_u32(sB) + kk * 2048, 8192)
                                     : sdesc_sw128(smem_u32(sB) + kk * 32);
            mma_bf16(tmem, ad, bd, idesc, kk > 0);
        }
        mma_commit(bar_mma);
    }
    if (ok) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar_mma, 0))
            if (clock64() - t0 > 2000000000LL) { ok = false; break; }
    }
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
        float r[32];
        const int row = warp * 32 + lane;
        for (int cb = 0; cb < N / 32; ++cb) {
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + cb * 32, r);
            for (int i = 0; i < 32; ++i) D[row * N + cb * 32 + i] = r[i];
        }
    } else if (lane == 0) {
        atomicExch(status, 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_mma(const void* A, const void* B, float* D, int N, int flags,
                                       int* status, void* stream) {
    using namespace kda;
    if (!A || !B || !D || !status || (N != 64 && N != 128) || flags < 0 || flags > 7)
        return KDA_ERR_INVALID_ARG;
    const bool a_mn = (flags >> 1) & 1, b_mn = (flags >> 2) & 1;
    if ((a_mn || b_mn) && !(flags & 1)) return KDA_ERR_INVALID_ARG;  // MN-major needs TMA
    CUtensorMap ma, mb;
    // A: [128 m][64 k] (K-major) or [64 k][128 m] (MN-major); B likewise with N.
    const bool okA = a_mn ? make_map_bf16(&ma, A, 64, 128, 64, 64)
                          : make_map_bf16(&ma, A, 128, 64, 64, 128);
    const bool okB = b_mn ? make_map_bf16(&mb, B, 64, N, 64, 64)
                          : make_map_bf16(&mb, B, N, 64, 64, N);
    if (!okA || !okB) return KDA_ERR_CUDA;
    const int smem = 147456 + 64 + 1024;
    if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        ma, mb, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D, N,
        flags, status);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
