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
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

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


// ------------------------------------------------------------------------------------------
// Bulk-copy pipeline for bf16 records of d = 128 (full record 67,840 B: S fp32 [128][128] and
// the window; INT8 record 19,200 B: scales, codes, window; neither needs padding) in pools of
// pages of at least 4 KiB.  One persistent CTA per SM walks the head records.
//   - A producer warp bulk-loads source records (split at page boundaries) into a ring of
//     source slots and bulk-stores converted records from a ring of destination slots.  The
//     page ids of the next item are read into registers one step ahead, so their global
//     reads overlap the current step.  A store's read-out of shared memory is waited for only
//     when its destination slot is needed again, two items later.
//   - Sixteen compute warps convert one item at a time from its source slot into its
//     destination slot: four threads per row of S, 32 consecutive values each (a row's
//     max-abs is a reduction over its four threads).
// Quantising: 2 source slots (67,840 B) and 2 destination slots (19,200 B); dequantising: 3
// source slots (19,200 B) and 2 destination slots (67,840 B).  The codes are those of the
// per-record kernels above, bit for bit: the division goes through the reciprocal where that
// provably gives the same integer (see below), through the IEEE division elsewhere.
constexpr int kQtCompute = 512;
constexpr int kQtThreads = kQtCompute + 32;
constexpr uint32_t kQtFull = 67840, kQtQ8 = 19200;
template <bool QUANT> struct QtGeom {
    static constexpr int NS = QUANT ? 2 : 3, ND = 2;
    static constexpr uint32_t SB = QUANT ? kQtFull : kQtQ8, DB = QUANT ? kQtQ8 : kQtFull;
    static constexpr uint32_t DST0 = NS * SB, MISC = DST0 + ND * DB, SMEM = MISC + 256;
    static_assert(SB % 128 == 0 && DB % 128 == 0 && SMEM <= 227 * 1024, "INT8 pipeline shared memory");
};

// Page index of in-object byte offset `off` (below 4 GiB): a shift for power-of-two page
// sizes, otherwise the high half of off * ceil(2^32 / page_bytes) corrected by one compare.
__device__ __forceinline__ uint32_t qt_page_of(const PoolView &v, uint32_t off) {
    if (v.page_shift >= 0) return off >> v.page_shift;
    uint32_t q = __umulhi(off, v.page_magic);
    if ((uint64_t)q * (uint64_t)v.page_bytes > off) --q;
    return q;
}

// Max over the four threads of a row (lanes 4 i .. 4 i + 3).
__device__ __forceinline__ float quad_max(float x) {
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
    return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

// One row quarter: 32 fp32 values (8 x 16 B, read in a rotated order so that the four
// threads of a row and the eight rows of a warp spread over all banks) -> 32 codes.
__device__ __forceinline__ void load_quarter(const float *row, int qq, int rot, float4 (&x)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = reinterpret_cast<const float4 *>(row)[qq * 8 + ((k + rot) & 7)];
}

__device__ __forceinline__ void quant_quarter(const float4 (&x)[8], uint8_t *crow, int qq, int rot, float *scale_out) {
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w))));
    m = quad_max(m);
    const float sc = __fdiv_rn(m, 127.f);
    // code = rint(RN(x / sc)) through the correctly rounded reciprocal, with Ziv's rounding
    // test: y = RN(x RN(1/sc)) lies within 127 * 2^-23 + 2^-18 < 2^-14 of RN(x / sc)
    // (|x / sc| <= 127), so rint(y) is that integer unless y is within 2^-14 of a
    // half-integer.  Such values, and rows whose reciprocal is not finite, take the IEEE
    // division; the branch is taken per warp and only when a lane needs it.
    const float rs = __frcp_rn(sc);
    const bool fast_row = sc > 0.f && isfinite(rs);
    bool near = !fast_row && sc > 0.f;
    auto pack4 = [](int q0, int q1, int q2, int q3) {
        auto c = [](int q) { return (uint32_t)((q > 127 ? 127 : (q < -127 ? -127 : q)) & 0xff); };
        return c(q0) | (c(q1) << 8) | (c(q2) << 16) | (c(q3) << 24);
    };
    // Rounding by the magic number 1.5 * 2^23: for |y| < 2^22, t = RN(y + 1.5 * 2^23) is y
    // rounded to the nearest integer (ties to even) plus 1.5 * 2^23, so the low byte of t's bits
    // is that integer's two's complement byte and t - 1.5 * 2^23 is the integer itself (exact).
    // Here |y| <= 127 (1 + 2^-23), so the code needs no clamp.
    constexpr float kMagic = 12582912.f;
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float xs[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
        uint32_t word = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float y = __fmul_rn(xs[u], rs);
            const float t = __fadd_rn(y, kMagic);
            const float d = __fsub_rn(y, __fsub_rn(t, kMagic));   // y - rint(y), in [-0.5, 0.5]
            near = near || fabsf(d) > 0.5f - 0x1p-14f;
            word |= (__float_as_uint(t) & 0xffu) << (8 * u);
        }
        w[k] = fast_row ? word : 0u;
    }
    if (__any_sync(0xffffffffu, near) && sc > 0.f) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            w[k] = pack4(__float2int_rn(__fdiv_rn(x[k].x, sc)), __float2int_rn(__fdiv_rn(x[k].y, sc)),
                         __float2int_rn(__fdiv_rn(x[k].z, sc)), __float2int_rn(__fdiv_rn(x[k].w, sc)));
    }
    // element k * 4 + u of the quarter goes to byte qq * 32 + k * 4 + u of the row, in the same
    // rotated order as the loads
#pragma unroll
    for (int k = 0; k < 8; ++k) reinterpret_cast<uint32_t *>(crow)[qq * 8 + ((k + rot) & 7)] = w[k];
    if (scale_out) *scale_out = sc;
}

// One row quarter back: 32 codes (read first, rotated order) and the row's scale -> 32 fp32
// values.
__device__ __forceinline__ void load_codes(const uint8_t *crow, int qq, int rot, uint32_t (&c8)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) c8[k] = reinterpret_cast<const uint32_t *>(crow)[qq * 8 + ((k + rot) & 7)];
}

__device__ __forceinline__ void dequant_quarter(const uint32_t (&c8)[8], float sc, float *row, int qq, int rot) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int w = qq * 8 + ((k + rot) & 7);
        const uint32_t c = c8[k];
        float4 v;
        v.x = (float)(signed char)(c & 0xff) * sc;
        v.y = (float)(signed char)((c >> 8) & 0xff) * sc;
        v.z = (float)(signed char)((c >> 16) & 0xff) * sc;
        v.w = (float)(signed char)(c >> 24) * sc;
        reinterpret_cast<float4 *>(row)[w] = v;
    }
}

template <bool QUANT>
__global__ void __launch_bounds__(kQtThreads, 1) q8_tma_kernel(Q8Args a) {
    using G = QtGeom<QUANT>;
    constexpr int D = 128, NS = G::NS, ND = G::ND;
    extern __shared__ __align__(128) uint8_t sm[];
    volatile int *valid = reinterpret_cast<volatile int *>(sm + G::MISC);        // [NS] per source slot
    volatile int *err = reinterpret_cast<volatile int *>(sm + G::MISC + 16);
    volatile int *go = reinterpret_cast<volatile int *>(sm + G::MISC + 20);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + G::MISC + 32);            // [NS] source loaded (tx)
    uint64_t *sfree = full + NS;                                                 // [NS] source read by compute
    uint64_t *dfull = sfree + NS;                                                // [ND] destination written
    uint64_t *dfree = dfull + ND;                                                // [ND] destination read by its store
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.n * a.H;
    const PoolView &sv = QUANT ? a.full : a.q8, &dv = QUANT ? a.q8 : a.full;
    const int32_t *spl = QUANT ? a.full_pages : a.q8_pages, *dpl = QUANT ? a.q8_pages : a.full_pages;
    if (tid == 0) {
        for (int i = 0; i < 2 * NS + 2 * ND; ++i) ptx::mbar_init(&full[i], 1);
        *err = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kQtCompute / 32) {
        // ------------------------------------------------------------------ producer
        // Page ids of an item's two lists live in the warp's registers (lane i: ids i and
        // i + 32); ids from 64 on are read from global memory where needed.
        constexpr int kIds = 2;
        struct Ids { int32_t s[kIds], d[kIds]; };
        auto lists = [&](int m, const int32_t *&sp, const int32_t *&dp) {
            const int obj = (blockIdx.x + m * gridDim.x) / a.H;
            sp = spl + (int64_t)obj * sv.pages_per_object;
            dp = dpl + (int64_t)obj * dv.pages_per_object;
        };
        auto fetch_ids = [&](int m, Ids &x) {
            const int32_t *sp, *dp;
            lists(m, sp, dp);
#pragma unroll
            for (int u = 0; u < kIds; ++u) {
                const int i = lane + 32 * u;
                x.s[u] = i < sv.pages_per_object ? sp[i] : 0;
                x.d[u] = i < dv.pages_per_object ? dp[i] : 0;
            }
        };
        auto ids_ok = [&](int m, const Ids &x) {
            bool ok = true;
#pragma unroll
            for (int u = 0; u < kIds; ++u)
                ok = ok && (uint32_t)x.s[u] < (uint32_t)sv.num_pages && (uint32_t)x.d[u] < (uint32_t)dv.num_pages;
            const int32_t *sp, *dp;
            lists(m, sp, dp);
            for (int i = lane + 32 * kIds; i < sv.pages_per_object; i += 32) ok = ok && (uint32_t)sp[i] < (uint32_t)sv.num_pages;
            for (int i = lane + 32 * kIds; i < dv.pages_per_object; i += 32) ok = ok && (uint32_t)dp[i] < (uint32_t)dv.num_pages;
            return __all_sync(0xffffffffu, ok);
        };
        // The record of head hh, piece by piece (at most one piece per page it touches): the whole
        // warp walks the pieces, the page id comes from the registers, lane 0 issues the copy.
        auto pieces = [&](const PoolView &v, const int32_t (&ids)[kIds], const int32_t *list, int hh, uint32_t bytes,
                          auto &&fn) {
            const uint32_t PB = (uint32_t)v.page_bytes;
            uint32_t off = (uint32_t)(hh * v.rec_bytes), at = 0;
            while (at < bytes) {
                const uint32_t pi = qt_page_of(v, off), in = off - pi * PB;
                const uint32_t len = bytes - at < PB - in ? bytes - at : PB - in;
                int32_t id = __shfl_sync(0xffffffffu, pi < 32 ? ids[0] : ids[1], pi & 31);
                if (pi >= 64) id = list[pi];
                if (lane == 0) fn(v.base + (uint64_t)id * v.page_bytes + in, at, len);
                off += len;
                at += len;
            }
        };
        Ids cur, nxt, prev;
        int dmask = 0;   // bit b: destination slot b holds a converted record to store
        int n = 0;
        if (blockIdx.x < total) fetch_ids(0, cur);
        for (;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int bs = n % NS;
            if (item + (int)gridDim.x < total) fetch_ids(n + 1, nxt);   // overlaps this step
            const bool ok = ids_ok(n, cur);
            // load item n once compute has read the item that used its source slot
            int stop = 0;
            if (lane == 0 && (*err || (n >= NS && !ptx::mbar_wait(&sfree[bs], (uint32_t)(((n - NS) / NS) & 1), err))))
                stop = 1;
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            const int32_t *sp, *dp;
            lists(n, sp, dp);
            if (lane == 0) {
                valid[bs] = ok ? 1 : 0;
                if (!ok) {
                    flag_status(a.status, KDA_DEV_BAD_PAGE);
                    ptx::mbar_arrive(&full[bs]);
                } else {
                    ptx::mbar_arrive_expect_tx(&full[bs], G::SB);
                }
            }
            if (ok)
                pieces(sv, cur.s, sp, item % a.H, G::SB, [&](uint8_t *g, uint32_t at, uint32_t len) {
                    ptx::bulk_load(sm + bs * G::SB + at, g, len, &full[bs]);
                });
            // store item n - 1 once compute has written it; then the destination slot of item
            // n - 2 is free as soon as that older store has read it out
            if (n >= 1) {
                const int m = n - 1, bd = m % ND;
                if (lane == 0 && !ptx::mbar_wait(&dfull[bd], (uint32_t)((m / ND) & 1), err)) stop = 1;
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
                const int32_t *psp, *pdp;
                lists(m, psp, pdp);
                if ((dmask >> bd) & 1)
                    pieces(dv, prev.d, pdp, (blockIdx.x + m * gridDim.x) % a.H, G::DB, [&](uint8_t *g, uint32_t at, uint32_t len) {
                        ptx::bulk_store(g, sm + G::DST0 + bd * G::DB + at, len);
                    });
                if (lane == 0) {
                    ptx::bulk_commit();
                    ptx::bulk_wait_read1();
                    if (m >= 1) ptx::mbar_arrive(&dfree[(m - 1) % ND]);
                }
            }
            __syncwarp();
            dmask = ok ? (dmask | (1 << (n % ND))) : (dmask & ~(1 << (n % ND)));
            prev = cur;
            cur = nxt;
        }
        if (!*err && n >= 1) {
            // the last item goes out
            const int m = n - 1, bd = m % ND;
            int stop = 0;
            if (lane == 0 && !ptx::mbar_wait(&dfull[bd], (uint32_t)((m / ND) & 1), err)) stop = 1;
            if (!__shfl_sync(0xffffffffu, stop, 0)) {
                const int32_t *psp, *pdp;
                lists(m, psp, pdp);
                if ((dmask >> bd) & 1)
                    pieces(dv, prev.d, pdp, (blockIdx.x + m * gridDim.x) % a.H, G::DB, [&](uint8_t *g, uint32_t at, uint32_t len) {
                        ptx::bulk_store(g, sm + G::DST0 + bd * G::DB + at, len);
                    });
                if (lane == 0) ptx::bulk_commit();
            }
        }
        if (lane == 0) {
            ptx::bulk_wait0();
            if (*err) {
                // leave no load in flight
                for (int m = n - NS < 0 ? 0 : n - NS; m < n; ++m) {
                    uint32_t k = 0;
                    while (!ptx::mbar_try_wait(&full[m % NS], (uint32_t)((m / NS) & 1)) && k < ptx::kSpinLimit) ++k;
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ compute
        // full record: S fp32 at 0, window at D*D*4; INT8 record: scales at 0, codes at 4 D,
        // window at 4 D + D*D
        constexpr uint32_t WF = D * D * 4, WQ = 4 * D + D * D, WBYTES = 9 * D * 2;
        const int r = tid >> 2, qq = tid & 3, rot = r & 7;   // row of S, quarter of the row
        for (int n = 0;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int bs = n % NS, bd = n % ND;
            if (tid == 0) {
                bool okw = ptx::mbar_wait(&full[bs], (uint32_t)((n / NS) & 1), err);
                if (okw && n >= ND) okw = ptx::mbar_wait(&dfree[bd], (uint32_t)(((n - ND) / ND) & 1), err);
                *go = (okw && !*err) ? 1 : 0;
            }
            tcx::named_bar(1, kQtCompute);
            if (!*go) break;
            const uint8_t *src = sm + bs * G::SB;
            uint8_t *dst = sm + G::DST0 + bd * G::DB;
            // every thread first takes its part of the source into registers; the source slot is
            // then released, so that the next load into it overlaps the conversion
            const bool vld = valid[bs] != 0;
            float4 x[8];
            uint32_t c8[8];
            float sc = 0.f;
            uint4 win = make_uint4(0, 0, 0, 0);
            if (vld) {
                if (QUANT) {
                    load_quarter(reinterpret_cast<const float *>(src) + r * D, qq, rot, x);
                    if (tid < WBYTES / 16) win = reinterpret_cast<const uint4 *>(src + WF)[tid];
                } else {
                    sc = reinterpret_cast<const float *>(src)[r];
                    load_codes(src + 4 * D + r * D, qq, rot, c8);
                    if (tid < WBYTES / 16) win = reinterpret_cast<const uint4 *>(src + WQ)[tid];
                }
            }
            tcx::named_bar(1, kQtCompute);
            if (tid == 0) ptx::mbar_arrive(&sfree[bs]);
            if (vld) {
                if (QUANT) {
                    quant_quarter(x, dst + 4 * D + r * D, qq, rot, qq == 0 ? &sc : nullptr);
                    if (qq == 0) reinterpret_cast<float *>(dst)[r] = sc;
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(dst + WQ)[tid] = win;
                } else {
                    dequant_quarter(c8, sc, reinterpret_cast<float *>(dst) + r * D, qq, rot);
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(dst + WF)[tid] = win;
                }
                ptx::fence_proxy_async_smem();
            }
            tcx::named_bar(1, kQtCompute);
            if (tid == 0) ptx::mbar_arrive(&dfull[bd]);
        }
    }
    __syncthreads();
    if (*err && tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
}

bool q8_tma_applies(const Q8Args &a) {
    return a.d == 128 && a.dtype == KDA_BF16 && a.full.rec_bytes == (int64_t)kQtFull &&
           a.q8.rec_bytes == (int64_t)kQtQ8 && a.full.page_bytes >= 4096 && a.q8.page_bytes >= 4096;
}

template <bool QUANT>
cudaError_t launch_q8_tma(const Q8Args &a, cudaStream_t s) {
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(q8_tma_kernel<QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QtGeom<QUANT>::SMEM);
    if (e != cudaSuccess) return e;
    const int total = a.n * a.H;
    q8_tma_kernel<QUANT><<<(unsigned)(total < nsm ? total : nsm), kQtThreads, QtGeom<QUANT>::SMEM, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ckpt_quantize(const Q8Args &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    if (q8_tma_applies(a)) return launch_q8_tma<true>(a, s);
    const unsigned grid = (unsigned)(a.n * a.H);
    if (a.d == 128) quantize_kernel<128><<<grid, kQThreads, 0, s>>>(a);
    else if (a.d == 64) quantize_kernel<64><<<grid, kQThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_ckpt_dequantize(const Q8Args &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    if (q8_tma_applies(a)) return launch_q8_tma<false>(a, s);
    const unsigned grid = (unsigned)(a.n * a.H);
    if (a.d == 128) dequantize_kernel<128><<<grid, kQThreads, 0, s>>>(a);
    else if (a.d == 64) dequantize_kernel<64><<<grid, kQThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace kda
