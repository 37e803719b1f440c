// Chunked varlen KDA prefill on CUDA cores in fp32 (the path for fp32 inputs).
//
// One CTA runs one (sequence, head) through its chunks of 64 tokens, aligned to absolute
// positions.  Within a chunk of rows r = 0..63 (padding rows outside the sequence act as
// identity tokens: alpha = 1, beta = 0, k = q = v = 0):
//   conv      xbar_r = sum_j w_j x_{r-3+j} for the q | k | v channels (window from the
//             previous chunk, the restored state, or zeros)
//   decay     gamma_r = prod_{s<=r} alpha_s (per key channel), qt = gamma q, kt = gamma k,
//             kh = k / gamma, kb = gamma_C kh
//   Gram      A[r][s] = beta_r kt_r . kh_s (s < r),   P[r][s] = qt_r . kh_s (s <= r)
//   write     (I + A) W = Diag(beta) (V - Kt S)        (forward substitution)
//   read      O = Qt S + P W
//   advance   S <- Diag(gamma_C) S + Kb^T W
// This is the token recurrence S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T,
// o_t = S_t^T q_t ("Lesson 01 · Architecture map", §两种 Attention，两种状态) grouped into
// chunks: the chunk acts on S as one affine map M_C S + b_C ("KIMI K3 경량 복제에서 본 KDA의
// AI 인프라 과제", §0x01 1.3), here with M_C = Diag(gamma_C) - Kb^T (I+A)^{-1} Diag(beta) Kt
// and b_C = Kb^T (I+A)^{-1} Diag(beta) V.
//
// At a chunk end equal to a listed checkpoint position the record (S fp32, then the last 3
// raw tokens) is written into that checkpoint's pages; the final state goes to the
// sequence's active object ("Cache de préfixe hybride KDA–MLA", §Le fonctionnement du
// prefill and §Les checkpoints sont en lecture seule).
//
// The decay factorisation divides by gamma; it is exact in fp32 as long as the product of
// alpha over one chunk stays at or above 2^-100 (kMinChunkDecay) in every channel.  A chunk
// below that sets KDA_DEV_RANGE.
#include "common.cuh"

namespace kda {
namespace {

constexpr int kSimtThreads = 256;

template <int D>
struct SimtSmem {
    static constexpr int C = kChunk;
    static constexpr int LD = D + 1;      // padded row stride of q / k / kh tiles
    static constexpr int CP = C + 1;      // padded row stride of A / P
    static constexpr int NI = kSimtThreads / D;
    static constexpr int RB = 16;         // rows per reduction block
    static constexpr int q_off = 0;
    static constexpr int k_off = q_off + C * LD;
    static constexpr int kh_off = k_off + C * LD;
    static constexpr int v_off = kh_off + C * LD;
    static constexpr int g_off = v_off + C * D;
    static constexpr int A_off = g_off + C * D;
    static constexpr int P_off = A_off + C * CP;
    static constexpr int red_off = P_off + C * CP;
    static constexpr int halo_off = red_off + NI * RB * D;
    static constexpr int gC_off = halo_off + kWin * 3 * D;
    static constexpr int b_off = gC_off + D;
    static constexpr int total = b_off + C;
    static constexpr size_t bytes = sizeof(float) * (size_t)total;
};

// Write S (registers, this thread's column j and rows [i0, i0+RPT)) and the window into a
// head record reached through `pages`.
template <int D, typename T, int RPT>
__device__ void write_record(const PoolView &pv, const int32_t *pages, uint64_t rec,
                             const float (&S)[RPT], int i0, int j, const float *halo,
                             int32_t *status) {
#pragma unroll
    for (int ii = 0; ii < RPT; ++ii) {
        float *p = reinterpret_cast<float *>(
            obj_addr(pv, pages, rec + ((uint64_t)(i0 + ii) * D + j) * 4, status));
        if (p) *p = S[ii];
    }
    const uint64_t wo = rec + (uint64_t)D * D * 4;
    for (int e = threadIdx.x; e < kWin * 3 * D; e += kSimtThreads) {
        T *p = reinterpret_cast<T *>(obj_addr(pv, pages, wo + (uint64_t)e * sizeof(T), status));
        if (p) st_elem(p, halo[e]);
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(kSimtThreads, 1) prefill_simt_kernel(PrefillArgs a) {
    using L = SimtSmem<D>;
    constexpr int C = kChunk, LD = L::LD, CP = L::CP, NI = L::NI, RB = L::RB;
    constexpr int RPT = D / NI;            // rows of S held by one thread
    constexpr int C3 = 3 * D;
    extern __shared__ float sm[];
    float *qs = sm + L::q_off, *ks = sm + L::k_off, *kh = sm + L::kh_off;
    float *vs = sm + L::v_off, *gs = sm + L::g_off, *As = sm + L::A_off, *Ps = sm + L::P_off;
    float *red = sm + L::red_off, *halo = sm + L::halo_off, *gC = sm + L::gC_off, *bs = sm + L::b_off;

    const int tid = threadIdx.x;
    const int h = blockIdx.x % a.H, sq = blockIdx.x / a.H;
    const SeqMeta m = a.seqs[sq];
    const int j = tid % D, part = tid / D, i0 = part * RPT;
    const int H = a.H;
    const uint64_t rec = (uint64_t)h * (uint64_t)a.pool.rec_bytes;
    const int32_t *act_pages = a.pages + m.active_off;

    const T *qg = static_cast<const T *>(a.q), *kg = static_cast<const T *>(a.k);
    const T *vg = static_cast<const T *>(a.v), *ag = static_cast<const T *>(a.alpha);
    const T *bg = static_cast<const T *>(a.beta);
    T *og = static_cast<T *>(a.o);

    // Initial state and window.
    float S[RPT];
    if (m.has_init) {
#pragma unroll
        for (int ii = 0; ii < RPT; ++ii) {
            const float *p = reinterpret_cast<const float *>(
                obj_addr(a.pool, act_pages, rec + ((uint64_t)(i0 + ii) * D + j) * 4, a.status));
            S[ii] = p ? *p : 0.f;
        }
        const uint64_t wo = rec + (uint64_t)D * D * 4;
        for (int e = tid; e < kWin * C3; e += kSimtThreads) {
            const T *p = reinterpret_cast<const T *>(obj_addr(a.pool, act_pages, wo + (uint64_t)e * sizeof(T), a.status));
            halo[e] = p ? ld_elem(p) : 0.f;
        }
    } else {
#pragma unroll
        for (int ii = 0; ii < RPT; ++ii) S[ii] = 0.f;
        for (int e = tid; e < kWin * C3; e += kSimtThreads) halo[e] = 0.f;
    }
    __syncthreads();

    const int64_t start = m.start_pos, end = m.start_pos + m.len;
    int nck = 0;
    const int64_t c_first = start / C;
    const int64_t c_last = m.len > 0 ? (end - 1) / C : c_first - 1;
    for (int64_t c = c_first; c <= c_last; ++c) {
        const int64_t abs0 = c * C;
        const int r_first = start > abs0 ? (int)(start - abs0) : 0;
        const int r_end = end - abs0 < C ? (int)(end - abs0) : C;
        const int64_t row0 = (int64_t)m.tok_begin + (abs0 - start);   // packed row of chunk row 0

        // 1. The chunk's raw rows into the tiles in one coalesced pass (rows outside the
        //    sequence read as zeros, their alpha as one), then the conv in place, each thread
        //    walking a channel down the chunk with the last three raw values in registers, and
        //    the cumulative decay in place over the alpha tile.
        for (int e = tid; e < C * C3; e += kSimtThreads) {
            const int r = e / C3, ch = e % C3, which = ch / D, cc = ch % D;
            const T *src = which == 0 ? qg : (which == 1 ? kg : vg);
            float *dst = which == 0 ? qs : (which == 1 ? ks : vs);
            const int ld = which == 2 ? D : LD;
            dst[r * ld + cc] = (r >= r_first && r < r_end) ? ld_elem(src + ((row0 + r) * H + h) * D + cc) : 0.f;
        }
        for (int e = tid; e < C * D; e += kSimtThreads) {
            const int r = e / D, i = e % D;
            gs[r * D + i] = (r >= r_first && r < r_end) ? ld_elem(ag + ((row0 + r) * H + h) * D + i) : 1.f;
        }
        if (tid < C) bs[tid] = (tid >= r_first && tid < r_end) ? ld_elem(bg + (row0 + tid) * H + h) : 0.f;
        __syncthreads();
        for (int col = tid; col < C3 + D; col += kSimtThreads) {
            if (col < C3) {
                const int ch = col, which = ch / D, cc = ch % D;
                const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ((int64_t)h * C3 + ch) * 4);
                float p0 = halo[ch], p1 = halo[C3 + ch], p2 = halo[2 * C3 + ch];
                float *dst = which == 0 ? qs : (which == 1 ? ks : vs);
                const int ld = which == 2 ? D : LD;
                for (int r = r_first; r < r_end; ++r) {
                    const float x = dst[r * ld + cc];
                    dst[r * ld + cc] = w.x * p0 + w.y * p1 + w.z * p2 + w.w * x;
                    p0 = p1; p1 = p2; p2 = x;
                }
                halo[ch] = p0; halo[C3 + ch] = p1; halo[2 * C3 + ch] = p2;
            } else {
                const int i = col - C3;
                float g = 1.f;
                for (int r = 0; r < C; ++r) {
                    g *= gs[r * D + i];
                    gs[r * D + i] = g;
                }
                gC[i] = g;
                if (!(g >= kMinChunkDecay)) flag_status(a.status, KDA_DEV_RANGE);   // kh = k / gamma reaches 1 / g
            }
        }
        __syncthreads();
        // 3. decay-scaled copies.
        for (int e = tid; e < C * D; e += kSimtThreads) {
            const int r = e / D, i = e % D;
            const float g = gs[r * D + i];
            const float kk = ks[r * LD + i];
            qs[r * LD + i] *= g;
            ks[r * LD + i] = kk * g;
            kh[r * LD + i] = kk / g;
        }
        __syncthreads();
        // 4. A = Diag(beta) strict_lower(Kt Kh^T), P = lower(Qt Kh^T); thread tile 4 x 4,
        //    rows tr + 16 a, columns ts + 16 b.
        {
            const int tr = tid / 16, ts = tid % 16;
            float accA[4][4], accP[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) { accA[x][y] = 0.f; accP[x][y] = 0.f; }
            for (int i = 0; i < D; ++i) {
                float kr[4], qr[4], hs[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    kr[x] = ks[(tr + 16 * x) * LD + i];
                    qr[x] = qs[(tr + 16 * x) * LD + i];
                    hs[x] = kh[(ts + 16 * x) * LD + i];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        accA[x][y] = fmaf(kr[x], hs[y], accA[x][y]);
                        accP[x][y] = fmaf(qr[x], hs[y], accP[x][y]);
                    }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int r = tr + 16 * x, s = ts + 16 * y;
                    As[r * CP + s] = s < r ? bs[r] * accA[x][y] : 0.f;
                    Ps[r * CP + s] = s <= r ? accP[x][y] : 0.f;
                }
        }
        __syncthreads();
        // 5. kb = gamma_C kh (kh no longer needed as such).
        for (int e = tid; e < C * D; e += kSimtThreads) {
            const int r = e / D, i = e % D;
            kh[r * LD + i] *= gC[i];
        }
        // 6. R = Diag(beta)(V - Kt S) in place of V, 16 rows at a time.
        for (int rb = 0; rb < C; rb += RB) {
            float pr[RB];
#pragma unroll
            for (int x = 0; x < RB; ++x) pr[x] = 0.f;
#pragma unroll
            for (int ii = 0; ii < RPT; ++ii) {
                const float sv = S[ii];
#pragma unroll
                for (int x = 0; x < RB; ++x) pr[x] = fmaf(ks[(rb + x) * LD + i0 + ii], sv, pr[x]);
            }
#pragma unroll
            for (int x = 0; x < RB; ++x) red[(part * RB + x) * D + j] = pr[x];
            __syncthreads();
            for (int e = tid; e < RB * D; e += kSimtThreads) {
                const int x = e / D, jj = e % D;
                float acc = 0.f;
#pragma unroll
                for (int pp = 0; pp < NI; ++pp) acc += red[(pp * RB + x) * D + jj];
                const int r = rb + x;
                vs[r * D + jj] = bs[r] * (vs[r * D + jj] - acc);
            }
            __syncthreads();
        }
        // 7. forward substitution (I + A) W = R, in place, in blocks of RB rows: a block's rows
        //    first take the terms of all earlier rows (split over the NI parts, summed through
        //    `red`), then part 0 solves within the block, one column per thread.
        for (int rb = 0; rb < C; rb += RB) {
            if (rb > 0) {
                float pr[RB];
#pragma unroll
                for (int x = 0; x < RB; ++x) pr[x] = 0.f;
                for (int s2 = part; s2 < rb; s2 += NI) {
                    const float w = vs[s2 * D + j];
#pragma unroll
                    for (int x = 0; x < RB; ++x) pr[x] = fmaf(As[(rb + x) * CP + s2], w, pr[x]);
                }
#pragma unroll
                for (int x = 0; x < RB; ++x) red[(part * RB + x) * D + j] = pr[x];
                __syncthreads();
                for (int e = tid; e < RB * D; e += kSimtThreads) {
                    const int x = e / D, jj = e % D;
                    float acc = 0.f;
#pragma unroll
                    for (int pp = 0; pp < NI; ++pp) acc += red[(pp * RB + x) * D + jj];
                    vs[(rb + x) * D + jj] -= acc;
                }
                __syncthreads();
            }
            if (part == 0) {
                for (int r = rb + 1; r < rb + RB; ++r) {
                    float w = vs[r * D + j];
                    for (int s2 = rb; s2 < r; ++s2) w = fmaf(-As[r * CP + s2], vs[s2 * D + j], w);
                    vs[r * D + j] = w;
                }
            }
            __syncthreads();
        }
        // 8. Y = Qt S into gs, 16 rows at a time.
        for (int rb = 0; rb < C; rb += RB) {
            float pr[RB];
#pragma unroll
            for (int x = 0; x < RB; ++x) pr[x] = 0.f;
#pragma unroll
            for (int ii = 0; ii < RPT; ++ii) {
                const float sv = S[ii];
#pragma unroll
                for (int x = 0; x < RB; ++x) pr[x] = fmaf(qs[(rb + x) * LD + i0 + ii], sv, pr[x]);
            }
#pragma unroll
            for (int x = 0; x < RB; ++x) red[(part * RB + x) * D + j] = pr[x];
            __syncthreads();
            for (int e = tid; e < RB * D; e += kSimtThreads) {
                const int x = e / D, jj = e % D;
                float acc = 0.f;
#pragma unroll
                for (int pp = 0; pp < NI; ++pp) acc += red[(pp * RB + x) * D + jj];
                gs[(rb + x) * D + jj] = acc;
            }
            __syncthreads();
        }
        // 9. O = Y + P W for the valid rows.
        for (int r = part; r < C; r += NI) {
            if (r < r_first || r >= r_end) continue;
            float o = gs[r * D + j];
            for (int s = 0; s <= r; ++s) o = fmaf(Ps[r * CP + s], vs[s * D + j], o);
            st_elem(og + ((row0 + r) * H + h) * D + j, o);
        }
        // 10. S <- Diag(gamma_C) S + Kb^T W.
#pragma unroll
        for (int ii = 0; ii < RPT; ++ii) S[ii] *= gC[i0 + ii];
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
            const float w = vs[r * D + j];
            const float *kr = kh + r * LD + i0;
#pragma unroll
            for (int ii = 0; ii < RPT; ++ii) S[ii] = fmaf(kr[ii], w, S[ii]);
        }
        // 11. checkpoints ending at this chunk.
        const int64_t cend = abs0 + r_end;
        while (nck < m.ckpt_count) {
            const CkptMeta ck = a.ckpts[m.ckpt_begin + nck];
            if (ck.pos > cend) break;
            if (ck.pos == cend)
                write_record<D, T, RPT>(a.pool, a.pages + ck.pages_off, rec, S, i0, j, halo, a.status);
            else if (tid == 0)
                flag_status(a.status, KDA_DEV_BAD_META);
            ++nck;
        }
        __syncthreads();
    }
    if (nck != m.ckpt_count && tid == 0) flag_status(a.status, KDA_DEV_BAD_META);
    write_record<D, T, RPT>(a.pool, act_pages, rec, S, i0, j, halo, a.status);
}

template <int D, typename T>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t s) {
    using L = SimtSmem<D>;
    auto kern = prefill_simt_kernel<D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(a.nseq * a.H), kSimtThreads, L::bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s) {
    if (a.d == 128) return a.dtype == KDA_BF16 ? launch_t<128, __nv_bfloat16>(a, s) : launch_t<128, float>(a, s);
    if (a.d == 64) return a.dtype == KDA_BF16 ? launch_t<64, __nv_bfloat16>(a, s) : launch_t<64, float>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace kda
