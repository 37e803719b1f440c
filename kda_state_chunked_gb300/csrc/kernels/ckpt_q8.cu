// INT8 compressed checkpoints: quantise an active object into an INT8 checkpoint object, and
// dequantise an INT8 checkpoint into an active object.
//
// Checkpoints waiting in the cache may hold the recurrent state in INT8 while the small conv
// window keeps its native precision; the scale is symmetric, one per key channel, from the
// max-abs along the value channels; a hit is dequantised once into a fresh active slot and the
// recurrence continues in full precision ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제",
// §0x05 5.3 and §0x06 6.6).
//
// INT8 head record (records one after another in head order, as in a full object):
//     scale fp32 [d] | codes int8 [d][d] (row i = key channel) | window [3][3d] in dtype
// zero-padded to a multiple of 256 bytes.  scale_i = max_j |S[i][j]| / 127 and
// code = round-to-nearest-even(S[i][j] / scale_i) clamped to [-127, 127], both divisions
// IEEE fp32; a zero row has scale 0 and codes 0; dequantisation is code * scale_i.
//
// One CTA per head record; warp w handles rows w, w + 8, ... of S, four at a time with the four
// loads issued before any is processed.  A row's max-abs is
// a warp shuffle reduction and every lane handles d/32 consecutive values (128-bit loads of the
// fp32 row at d = 128): both directions are one streaming pass over the two records.
#include "common.cuh"

namespace kda {
namespace {

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;
constexpr int kGroup = 4;                 // rows whose loads a warp keeps in flight together

template <int VEC> struct FVec;
template <> struct FVec<4> { using type = float4; };
template <> struct FVec<2> { using type = float2; };
template <int VEC> struct CVec;
template <> struct CVec<4> { using type = char4; };
template <> struct CVec<2> { using type = char2; };

// Logical byte `off` of an object through its page list (32-bit arithmetic: an object is far
// below 4 GiB), or nullptr with KDA_DEV_BAD_PAGE for a page id outside the pool.
__device__ __forceinline__ uint8_t *q_addr(const PoolView &pv, const int32_t *pages, uint32_t off, int32_t *status) {
    const uint32_t pb = (uint32_t)pv.page_bytes;
    // page sizes are usually powers of two: a shift instead of a division
    const uint32_t pi = (pb & (pb - 1)) == 0 ? off >> (__ffs(pb) - 1) : off / pb;
    const int32_t id = pages[pi];
    if ((uint32_t)id >= (uint32_t)pv.num_pages) {
        flag_status(status, KDA_DEV_BAD_PAGE);
        return nullptr;
    }
    return pv.base + (uint64_t)id * pv.page_bytes + (off - pi * pb);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Copy `bytes` (multiple of 16) from one object's logical offset to another's, 16 bytes per
// thread per step; zero-fill `zero` further bytes after the destination range.
__device__ void copy_units(const PoolView &sp, const int32_t *spg, uint32_t soff, const PoolView &dp,
                           const int32_t *dpg, uint32_t doff, uint32_t bytes, uint32_t zero, int32_t *status) {
    for (uint32_t x = threadIdx.x; x < (bytes + zero) / 16; x += kQThreads) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (x < bytes / 16) {
            const uint4 *s = reinterpret_cast<const uint4 *>(q_addr(sp, spg, soff + x * 16, status));
            if (s) v = *s;
        }
        uint4 *d = reinterpret_cast<uint4 *>(q_addr(dp, dpg, doff + x * 16, status));
        if (d) *d = v;
    }
}

// The object's page lists, staged in shared memory when they fit (every access translates
// through them); otherwise read from global memory.
constexpr int kListCap = 1024;

__device__ __forceinline__ void stage_lists(const Q8Args &a, int obj, int32_t *sf, int32_t *sq, const int32_t *&fpg,
                                            const int32_t *&qpg) {
    fpg = a.full_pages + (int64_t)obj * a.full.pages_per_object;
    qpg = a.q8_pages + (int64_t)obj * a.q8.pages_per_object;
    if (a.full.pages_per_object <= kListCap && a.q8.pages_per_object <= kListCap) {
        for (int i = threadIdx.x; i < a.full.pages_per_object; i += kQThreads) sf[i] = fpg[i];
        for (int i = threadIdx.x; i < a.q8.pages_per_object; i += kQThreads) sq[i] = qpg[i];
        __syncthreads();
        fpg = sf;
        qpg = sq;
    }
}

template <int D>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(Q8Args a) {
    constexpr int VEC = D / 32;
    using FV = typename FVec<VEC>::type;
    using CV = typename CVec<VEC>::type;
    __shared__ int32_t sf[kListCap], sq[kListCap];
    const int obj = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t *fpg, *qpg;
    stage_lists(a, obj, sf, sq, fpg, qpg);
    const uint32_t frec = (uint32_t)(h * a.full.rec_bytes), qrec = (uint32_t)(h * a.q8.rec_bytes);
    // rows in groups of kGroup: the group's loads are issued before any of it is processed
    constexpr int RPW = D / kQWarps;
#pragma unroll 1
    for (int k0 = 0; k0 < RPW; k0 += kGroup) {
    FV v[kGroup];
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        const int i = warp + (k0 + k) * kQWarps;
        const FV *src = reinterpret_cast<const FV *>(q_addr(a.full, fpg, frec + (uint32_t)(i * D + lane * VEC) * 4, a.status));
        v[k] = src ? __ldcs(src) : FV{};
    }
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        const int i = warp + (k0 + k) * kQWarps;
        const float *vf = reinterpret_cast<const float *>(&v[k]);
        float m = 0.f;
#pragma unroll
        for (int u = 0; u < VEC; ++u) m = fmaxf(m, fabsf(vf[u]));
        m = warp_max(m);
        const float scale = __fdiv_rn(m, 127.f);
        CV c;
        signed char *cc = reinterpret_cast<signed char *>(&c);
#pragma unroll
        for (int u = 0; u < VEC; ++u) {
            int q = scale > 0.f ? __float2int_rn(__fdiv_rn(vf[u], scale)) : 0;
            q = q > 127 ? 127 : (q < -127 ? -127 : q);
            cc[u] = (signed char)q;
        }
        CV *dst = reinterpret_cast<CV *>(q_addr(a.q8, qpg, qrec + 4 * D + (uint32_t)(i * D + lane * VEC), a.status));
        if (dst) __stcs(dst, c);
        if (lane == 0) {
            float *sd = reinterpret_cast<float *>(q_addr(a.q8, qpg, qrec + 4 * i, a.status));
            if (sd) *sd = scale;
        }
    }
    }
    // window, unchanged, then the record's zero padding
    const uint32_t wbytes = 9 * D * (a.dtype == KDA_BF16 ? 2 : 4);
    const uint32_t used = 4 * D + D * D + wbytes;
    copy_units(a.full, fpg, frec + D * D * 4, a.q8, qpg, qrec + 4 * D + D * D, wbytes,
               (uint32_t)a.q8.rec_bytes - used, a.status);
}

template <int D>
__global__ void __launch_bounds__(kQThreads) dequantize_kernel(Q8Args a) {
    constexpr int VEC = D / 32;
    using FV = typename FVec<VEC>::type;
    using CV = typename CVec<VEC>::type;
    __shared__ int32_t sf[kListCap], sq[kListCap];
    const int obj = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t *fpg, *qpg;
    stage_lists(a, obj, sf, sq, fpg, qpg);
    const uint32_t frec = (uint32_t)(h * a.full.rec_bytes), qrec = (uint32_t)(h * a.q8.rec_bytes);
    constexpr int RPW = D / kQWarps;
#pragma unroll 1
    for (int k0 = 0; k0 < RPW; k0 += kGroup) {
    float sc[kGroup];
    CV c[kGroup];
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        const int i = warp + (k0 + k) * kQWarps;
        const float *sp = reinterpret_cast<const float *>(q_addr(a.q8, qpg, qrec + 4 * i, a.status));
        sc[k] = sp ? *sp : 0.f;
        const CV *cp = reinterpret_cast<const CV *>(q_addr(a.q8, qpg, qrec + 4 * D + (uint32_t)(i * D + lane * VEC), a.status));
        c[k] = cp ? __ldcs(cp) : CV{};
    }
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
        const int i = warp + (k0 + k) * kQWarps;
        const signed char *cc = reinterpret_cast<const signed char *>(&c[k]);
        FV v;
        float *vf = reinterpret_cast<float *>(&v);
#pragma unroll
        for (int u = 0; u < VEC; ++u) vf[u] = (float)cc[u] * sc[k];
        FV *dst = reinterpret_cast<FV *>(q_addr(a.full, fpg, frec + (uint32_t)(i * D + lane * VEC) * 4, a.status));
        if (dst) __stcs(dst, v);
    }
    }
    const uint32_t wbytes = 9 * D * (a.dtype == KDA_BF16 ? 2 : 4);
    const uint32_t used = D * D * 4 + wbytes;
    copy_units(a.q8, qpg, qrec + 4 * D + D * D, a.full, fpg, frec + D * D * 4, wbytes,
               (uint32_t)a.full.rec_bytes - used, a.status);
}

}  // namespace

cudaError_t launch_ckpt_quantize(const Q8Args &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.n * a.H);
    if (a.d == 128) quantize_kernel<128><<<grid, kQThreads, 0, s>>>(a);
    else if (a.d == 64) quantize_kernel<64><<<grid, kQThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_ckpt_dequantize(const Q8Args &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.n * a.H);
    if (a.d == 128) dequantize_kernel<128><<<grid, kQThreads, 0, s>>>(a);
    else if (a.d == 64) dequantize_kernel<64><<<grid, kQThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace kda
