// Device helpers shared by the tensor-core prefill kernels: bf16 packing, named barriers,
// the tf32 mma.sync block products of the triangular solve, and warpgroup-uniform waits.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

#include "sm100_ptx.cuh"

namespace kda {
namespace tcx {

__device__ __forceinline__ uint32_t par(int lc) { return (uint32_t)((lc >> 1) & 1); }

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) { return f2_to_bf2(lo, hi); }

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Two-lane fp32 arithmetic (one instruction for a channel pair).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)),
          "l"(*reinterpret_cast<const uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D = A(16x8, row) * B(8x8, col) + D, tf32 in, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// fp32 64x64 solve scratch, XOR-swizzled so that mma.sync fragment loads avoid conflicts.
__device__ __forceinline__ int msc_idx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

// 16x16 block (bi, bj) product accumulate: acc(C-frag, 2 n-tiles) += M[bi,bk] * M[bk,bj].
__device__ __forceinline__ void blk_mma(float (&acc)[2][4], const float *M, int bi, int bk, int bj, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
        uint32_t a[4];
        const int r0 = bi * 16, c0 = bk * 16 + kt * 8;
        a[0] = to_tf32(M[msc_idx(r0 + g, c0 + t)]);
        a[1] = to_tf32(M[msc_idx(r0 + g + 8, c0 + t)]);
        a[2] = to_tf32(M[msc_idx(r0 + g, c0 + t + 4)]);
        a[3] = to_tf32(M[msc_idx(r0 + g + 8, c0 + t + 4)]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b[2];
            const int k0 = bk * 16 + kt * 8, n0 = bj * 16 + nt * 8;
            b[0] = to_tf32(M[msc_idx(k0 + t, n0 + g)]);
            b[1] = to_tf32(M[msc_idx(k0 + t + 4, n0 + g)]);
            mma_tf32(acc[nt], a, b);
        }
    }
}

__device__ __forceinline__ void blk_store(float *M, int bi, int bj, const float (&acc)[2][4], float scale, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int r0 = bi * 16, c0 = bj * 16 + nt * 8 + 2 * t;
        M[msc_idx(r0 + g, c0)] = scale * acc[nt][0];
        M[msc_idx(r0 + g, c0 + 1)] = scale * acc[nt][1];
        M[msc_idx(r0 + g + 8, c0)] = scale * acc[nt][2];
        M[msc_idx(r0 + g + 8, c0 + 1)] = scale * acc[nt][3];
    }
}

struct Shared {
    uint8_t *base;
    uint64_t *bar;
    volatile int *err;
    uint32_t *tmem;
};

__device__ __forceinline__ bool wait_bar(const Shared &s, int idx, uint32_t parity) {
    return ptx::mbar_wait(&s.bar[idx], parity, s.err);
}

// Warpgroup-uniform wait: thread 0 of the group polls (bounded), a named barrier hands the
// outcome to all 128 threads, so the whole group continues or stops together.
__device__ __forceinline__ bool wg_wait(const Shared &s, int idx, uint32_t parity, int wg_tid, int bar_id,
                                        volatile int *flag) {
    if (wg_tid == 0) *flag = ptx::mbar_wait(&s.bar[idx], parity, s.err) ? 1 : 0;
    named_bar(bar_id, 128);
    const bool ok = *flag != 0;
    named_bar(bar_id, 128);
    return ok;
}

// Warp-uniform wait: lane 0 polls (bounded) and broadcasts the outcome to the warp.
__device__ __forceinline__ bool warp_wait(const Shared &s, int idx, uint32_t parity) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait(&s.bar[idx], parity, s.err) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One arrival for the whole warp once every lane's earlier writes are ordered before it
// (barriers that count warps rather than threads).
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
}

}  // namespace tcx
}  // namespace kda
