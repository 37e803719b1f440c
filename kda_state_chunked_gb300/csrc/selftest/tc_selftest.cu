// Test-only library (libkda_selftest.so, loaded by the GPU tests, never by the product): a
// self-test of the tensor-core building blocks used by the prefill kernels: shared-memory
// operand layouts (128-byte swizzle, K-major and MN-major), the tcgen05 instruction and
// matrix descriptors, negate-A, accumulation, TMEM loads, and a TMA-loaded operand.
//
// D[128][N] = (neg ? -2 : 2) * A[128][K] * B[K][N] computed as two passes of K/16 MMAs
// (the second accumulating), A and B bf16 row-major in global memory, D fp32.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "../kernels/common.cuh"
#include "../kernels/sm100_ptx.cuh"

namespace kda {
namespace {

constexpr int kM = 128;

struct SelftestArgs {
    const __nv_bfloat16 *A;   // [128][K]
    const __nv_bfloat16 *B;   // [K][N]
    float *D;                 // [128][N]
    int K, N, a_mn, b_mn, neg, use_tma, a_tmem;
    int *err;
};

__global__ void __launch_bounds__(128, 1) mma_selftest_kernel(SelftestArgs a, const __grid_constant__ CUtensorMap tmA) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = ptx::smem_align1024(smem_raw);
    uint8_t *sA = sm;                        // up to 128 x 128 bf16 = 32 KiB
    uint8_t *sB = sm + 32768;                // up to 128 x 128 bf16 = 32 KiB
    __shared__ uint64_t bar_mma, bar_tma;
    __shared__ uint32_t tmem_base;
    __shared__ int err_s;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int K = a.K, N = a.N;
    if (tid == 0) {
        ptx::mbar_init(&bar_mma, 1);
        ptx::mbar_init(&bar_tma, 1);
        ptx::fence_mbar_init();
        err_s = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_base, 256);
        ptx::tmem_relinquish();
    }
    __syncthreads();
    // A operand into shared memory.
    if (a.use_tma) {
        // K-major A via TMA: boxes of 64 columns x 128 rows, one per 64-wide K block.
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(&bar_tma, (uint32_t)(kM * K * 2));
            for (int kb = 0; kb < K / 64; ++kb) ptx::tma_load_2d(sA + kb * (kM * 128), &tmA, &bar_tma, kb * 64, 0);
        }
    } else {
        for (int e = tid; e < kM * K; e += blockDim.x) {
            const int m = e / K, k = e % K;
            uint32_t off;
            if (a.a_mn) off = (m / 64) * (K * 128) + ptx::sw128_off(k, (m % 64) * 2);
            else off = (k / 64) * (kM * 128) + ptx::sw128_off(m, (k % 64) * 2);
            *reinterpret_cast<__nv_bfloat16 *>(sA + off) = a.A[e];
        }
    }
    for (int e = tid; e < K * N; e += blockDim.x) {
        const int k = e / N, n = e % N;
        uint32_t off;
        if (a.b_mn) off = (n / 64) * (K * 128) + ptx::sw128_off(k, (n % 64) * 2);
        else off = (k / 64) * (N * 128) + ptx::sw128_off(n, (k % 64) * 2);
        *reinterpret_cast<__nv_bfloat16 *>(sB + off) = a.B[e];
    }
    if (a.a_tmem) {
        // A into TMEM columns 128.. : thread m holds row m, bf16 pairs packed along K.
        __syncthreads();
        const int m = warp * 32 + (tid & 31);
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int c0 = 0; c0 < K / 2; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int k = 2 * (c0 + i);
                __nv_bfloat162 pr = __halves2bfloat162(a.A[(int64_t)m * K + k], a.A[(int64_t)m * K + k + 1]);
                v[i] = __uint_as_float(*reinterpret_cast<uint32_t *>(&pr));
            }
            if (c0 < K / 2) ptx::tmem_st32(tmem_base + lane_base + 128 + c0, v);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (a.use_tma && !ptx::mbar_wait(&bar_tma, 0, &err_s)) {
        if (tid == 0) atomicOr(a.err, 1);
    }
    ptx::tc_fence_after();
    if (tid == 0 && !err_s) {
        const uint32_t idesc = ptx::idesc_bf16(kM, N, a.a_mn, a.b_mn, a.neg);
        const uint32_t aBase = ptx::smem_u32(sA), bBase = ptx::smem_u32(sB);
        for (int pass = 0; pass < 2; ++pass) {
            for (int s = 0; s < K / 16; ++s) {
                uint64_t ad, bd;
                if (a.a_mn) ad = ptx::sdesc_sw128(aBase + s * 2048, K * 128, 1024);
                else ad = ptx::sdesc_sw128(aBase + (s / 4) * (kM * 128) + (s % 4) * 32, 16, 1024);
                if (a.b_mn) bd = ptx::sdesc_sw128(bBase + s * 2048, K * 128, 1024);
                else bd = ptx::sdesc_sw128(bBase + (s / 4) * (N * 128) + (s % 4) * 32, 16, 1024);
                if (a.a_tmem) ptx::mma_bf16_ta(tmem_base, tmem_base + 128 + s * 8, bd, idesc, (pass > 0 || s > 0) ? 1u : 0u);
                else ptx::mma_bf16(tmem_base, ad, bd, idesc, (pass > 0 || s > 0) ? 1u : 0u);
            }
        }
        ptx::mma_commit(&bar_mma);
    }
    __syncthreads();
    if (!err_s && !ptx::mbar_wait(&bar_mma, 0, &err_s)) {
        if (tid == 0) atomicOr(a.err, 2);
    }
    ptx::tc_fence_after();
    __syncthreads();
    if (!err_s) {
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            ptx::tmem_ld32(tmem_base + lane_base + (uint32_t)c0, v);
            ptx::tmem_wait_ld();
            const int m = warp * 32 + (tid & 31);
#pragma unroll
            for (int i = 0; i < 32; ++i) a.D[(int64_t)m * N + c0 + i] = v[i];
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem_base, 256);
}

}  // namespace

int encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows);

}  // namespace kda

// Entry point of the test-only library libkda_selftest.so (not part of libkda.so or its
// header): runs the self-test on device buffers and returns 0 or a negative setup error; the
// kernel's error bits go to err_dev.
extern "C" int kda_internal_mma_selftest(const void *A, const void *B, float *D, int K, int N, int a_mn, int b_mn,
                                         int neg, int use_tma, int *err_dev, void *stream) {
    using namespace kda;
    // use_tma == 2 selects an A operand read from TMEM instead of shared memory
    const int a_tmem = use_tma == 2 ? 1 : 0;
    if (a_tmem) use_tma = 0;
    if ((K != 64 && K != 128) || (N != 64 && N != 128) || !A || !B || !D || !err_dev) return -1;
    if ((use_tma || a_tmem) && a_mn) return -1;
    CUtensorMap tm;
    std::memset(&tm, 0, sizeof(tm));
    if (use_tma && encode_tmap_bf16_2d(&tm, A, (uint64_t)K, 128, (uint64_t)K * 2, 64, 128) != 0) return -3;
    SelftestArgs a{static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), D, K, N, a_mn,
                   b_mn, neg, use_tma, a_tmem, err_dev};
    const int smem = 65536 + 1024;
    auto kern = mma_selftest_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -4;
    kern<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(a, tm);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
