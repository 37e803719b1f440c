// Batched single-token KDA decode step over states gathered through a page table.
//
// Per (request, head): conv of the new token with the stored window (the window is shifted
// in place), then S' = Diag(alpha) S, w = beta (v - S'^T k), S = S' + k w^T, o = S^T q, with
// S written back in place.  The order (decay, delta write, read) follows "Lesson 01 ·
// Architecture map", §两种 Attention，两种状态; the fused conv + recurrent decode on the
// state indices follows "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" §0x08 8.2.2 and the
// block-table gather of "Chapitre 8 — Gestion nouvelle génération du cache KV" §8.1
// (PagedAttention: logical blocks mapped to physical pages through a table).
//
// The kernel is HBM-bound (about 0.84 flop per byte): each CTA streams one 64 KiB fp32
// state (d = 128) in and out once.  Warp w of 16 owns D/16 consecutive rows of S; lane l owns
// D/32 consecutive columns, so every row is one coalesced 512-byte (d = 128) access made
// of 128-bit loads, the state stays in registers between the two passes, the row
// reductions for S'^T k and S^T q are thread-local and one shared-memory pass combines
// the sixteen warps.  Sixteen warps per CTA and two CTAs per SM keep 64 KiB of state loads
// in flight per CTA while the other CTA computes.
#include "common.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;

template <int VEC> struct VecT;
template <> struct VecT<4> { using type = float4; };
template <> struct VecT<2> { using type = float2; };

template <int VEC>
__device__ __forceinline__ void vload(const uint8_t *p, float (&x)[VEC]) {
    using V = typename VecT<VEC>::type;
    const V t = __ldcs(reinterpret_cast<const V *>(p));
    const float *f = reinterpret_cast<const float *>(&t);
#pragma unroll
    for (int i = 0; i < VEC; ++i) x[i] = f[i];
}

template <int VEC>
__device__ __forceinline__ void vstore(uint8_t *p, const float (&x)[VEC]) {
    using V = typename VecT<VEC>::type;
    V t;
    float *f = reinterpret_cast<float *>(&t);
#pragma unroll
    for (int i = 0; i < VEC; ++i) f[i] = x[i];
    __stcs(reinterpret_cast<V *>(p), t);
}

template <int D, typename T>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeArgs a) {
    constexpr int C3 = 3 * D;
    constexpr int RPW = D / kDecWarps;   // rows of S per warp
    constexpr int VEC = D / 32;          // columns per lane
    __shared__ float xb[C3];             // post-conv q | k | v of the new token
    __shared__ float al[D];
    __shared__ float red[kDecWarps][D];
    __shared__ float wv[D];
    __shared__ float beta_s;
    __shared__ int ok_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int32_t *pages = a.state_pages + (int64_t)b * a.pool.pages_per_object;
    if (tid == 0) {
        ok_s = pages_ok(a.pool, pages);
        if (!ok_s) flag_status(a.status, KDA_DEV_BAD_PAGE);
    }
    __syncthreads();
    if (!ok_s) return;

    const uint64_t rec = (uint64_t)h * (uint64_t)a.pool.rec_bytes;
    const uint64_t win_off = rec + (uint64_t)D * D * 4;
    const int64_t tok = ((int64_t)b * a.H + h) * D;

    // Issue the state loads first: they are the bulk of the traffic.
    float s[RPW][VEC];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int i = warp * RPW + rr;
        const uint8_t *p = obj_addr(a.pool, pages, rec + ((uint64_t)i * D + lane * VEC) * 4, a.status);
        vload<VEC>(p, s[rr]);
    }

    // Conv of the new token against the stored window, then shift the window in place.
    const T *qp = static_cast<const T *>(a.q), *kp = static_cast<const T *>(a.k),
            *vp = static_cast<const T *>(a.v);
    for (int c = tid; c < C3; c += kDecThreads) {
        const T *src = c < D ? qp + tok + c : (c < 2 * D ? kp + tok + (c - D) : vp + tok + (c - 2 * D));
        const float x = ld_elem(src);
        const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ((int64_t)h * C3 + c) * 4);
        T *wp[kWin];
        float pv[kWin];
#pragma unroll
        for (int u = 0; u < kWin; ++u) {
            wp[u] = reinterpret_cast<T *>(obj_addr(a.pool, pages, win_off + ((uint64_t)u * C3 + c) * sizeof(T), a.status));
            pv[u] = ld_elem(wp[u]);
        }
        xb[c] = w.x * pv[0] + w.y * pv[1] + w.z * pv[2] + w.w * x;
        *wp[0] = *wp[1];
        *wp[1] = *wp[2];
        *wp[2] = *src;
    }
    const T *ap = static_cast<const T *>(a.alpha);
    for (int i = tid; i < D; i += kDecThreads) al[i] = ld_elem(ap + tok + i);
    if (tid == 0) beta_s = ld_elem(static_cast<const T *>(a.beta) + (int64_t)b * a.H + h);
    __syncthreads();

    // S' = Diag(alpha) S and the partial column sums of S'^T k over this warp's rows.
    float part[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) part[v] = 0.f;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int i = warp * RPW + rr;
        const float ai = al[i], ki = xb[D + i];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            s[rr][v] *= ai;
            part[v] = fmaf(ki, s[rr][v], part[v]);
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) red[warp][lane * VEC + v] = part[v];
    __syncthreads();
    for (int j = tid; j < D; j += kDecThreads) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) acc += red[w][j];
        wv[j] = beta_s * (xb[2 * D + j] - acc);
    }
    __syncthreads();

    // S = S' + k w^T, written back in place, and the partial sums of S^T q.
    float wl[VEC], po[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { wl[v] = wv[lane * VEC + v]; po[v] = 0.f; }
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int i = warp * RPW + rr;
        const float ki = xb[D + i], qi = xb[i];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            s[rr][v] = fmaf(ki, wl[v], s[rr][v]);
            po[v] = fmaf(qi, s[rr][v], po[v]);
        }
        uint8_t *p = obj_addr(a.pool, pages, rec + ((uint64_t)i * D + lane * VEC) * 4, a.status);
        vstore<VEC>(p, s[rr]);
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) red[warp][lane * VEC + v] = po[v];
    __syncthreads();
    T *op = static_cast<T *>(a.o);
    for (int j = tid; j < D; j += kDecThreads) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) acc += red[w][j];
        st_elem(op + tok + j, acc);
    }
}

template <int D, typename T>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s) {
    decode_kernel<D, T><<<(unsigned)(a.B * a.H), kDecThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (a.d == 128) return a.dtype == KDA_BF16 ? launch_decode_t<128, __nv_bfloat16>(a, s)
                                               : launch_decode_t<128, float>(a, s);
    if (a.d == 64) return a.dtype == KDA_BF16 ? launch_decode_t<64, __nv_bfloat16>(a, s)
                                              : launch_decode_t<64, float>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace kda
