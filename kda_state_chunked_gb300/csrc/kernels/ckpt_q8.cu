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
//   - A load warp bulk-loads source records (split at page boundaries) into a ring of source
//     slots, as far ahead as the ring allows: a slot is refilled as soon as the compute warps
//     have taken its record into registers.
//   - A store warp bulk-stores converted records from a ring of destination slots; a slot is
//     released once its store has read it out.
//   - Both read an item's page ids into registers two steps ahead, so those global reads
//     overlap the steps in between, and each checks its own list before using it.
//   - Sixteen compute warps convert one item at a time from its source slot into its
//     destination slot: four threads per row of S, 32 consecutive values each (a row's
//     max-abs is a reduction over its four threads).
// Quantising: 3 source slots (67,840 B) and 1 destination slot (19,200 B); dequantising: 3
// source slots (19,200 B) and 2 destination slots (67,840 B), with up to two stores in flight.
// For finite states the codes are those of the per-record kernels above, bit for bit: the
// division goes through the reciprocal where that provably gives the same integer (see below),
// through the IEEE division elsewhere.  (A state holding inf or NaN, which no valid recurrence
// produces, gets unspecified codes from either kernel.)
constexpr int kQtCompute = 512;
constexpr int kQtThreads = kQtCompute + 64;   // + load warp + store warp
constexpr uint32_t kQtFull = 67840, kQtQ8 = 19200;
template <bool QUANT> struct QtGeom {
    static constexpr int NS = 3, ND = QUANT ? 1 : 2;
    static constexpr uint32_t SB = QUANT ? kQtFull : kQtQ8, DB = QUANT ? kQtQ8 : kQtFull;
    static constexpr uint32_t DST0 = NS * SB, MISC = DST0 + ND * DB, SMEM = MISC + 256;
    static_assert(SB % 128 == 0 && DB % 128 == 0 && SMEM <= 227 * 1024, "INT8 pipeline shared memory");
    static_assert(NS <= 4 && ND <= 4, "slot flags: valid[4] at +0, dvalid[4] at +64, barriers from +128");
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

// Codes of the quarter into registers; returns the row's scale.
__device__ __forceinline__ float quant_quarter(const float4 (&x)[8], uint32_t (&w)[8]) {
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w))));
    m = quad_max(m);
    const float sc = __fdiv_rn(m, 127.f);
    // code = rint(RN(x / sc)) through the correctly rounded reciprocal, with Ziv's rounding
    // test.  With rs = RN(1/sc) and y = RN(x rs): |x rs - x/sc| <= |x/sc| 2^-24 < 2^-17
    // (|x/sc| <= 127 (1 + 2^-23)), and y and RN(x/sc) each lie within half an ulp of 64..128,
    // 2^-18, of x rs and x/sc.  So |y - RN(x/sc)| < 2^-16, and rint(y) is rint(RN(x/sc))
    // unless y is within 2^-16 of a half-integer.  Such values, and rows whose reciprocal is
    // not finite, take the IEEE division; the branch is taken per warp and only when a lane
    // needs it.
    const float rs = __frcp_rn(sc);
    const bool fast_row = sc > 0.f && isfinite(rs);
    auto pack4 = [](int q0, int q1, int q2, int q3) {
        auto c = [](int q) { return (uint32_t)((q > 127 ? 127 : (q < -127 ? -127 : q)) & 0xff); };
        return c(q0) | (c(q1) << 8) | (c(q2) << 16) | (c(q3) << 24);
    };
    // Rounding by the magic number 1.5 * 2^23: for |y| < 2^22, t = RN(y + 1.5 * 2^23) is y
    // rounded to the nearest integer (ties to even) plus 1.5 * 2^23, so the low byte of t's bits
    // is that integer's two's complement byte and t - 1.5 * 2^23 is the integer itself (exact).
    // Here |y| <= 127 (1 + 2^-23), so the code needs no clamp.  The arithmetic runs on value
    // pairs (one f32x2 instruction, each lane correctly rounded as the scalar one).
    constexpr float kMagic = 12582912.f;
    const float2 rs2 = make_float2(rs, rs), mg2 = make_float2(kMagic, kMagic);
    float dmax = 0.f;   // largest |y - rint(y)| of the quarter
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 ya = tcx::fmul2(make_float2(x[k].x, x[k].y), rs2);
        const float2 yb = tcx::fmul2(make_float2(x[k].z, x[k].w), rs2);
        const float2 ta = tcx::fadd2(ya, mg2), tb = tcx::fadd2(yb, mg2);
        const float2 da = tcx::fsub2(ya, tcx::fsub2(ta, mg2)), db = tcx::fsub2(yb, tcx::fsub2(tb, mg2));
        dmax = fmaxf(dmax, fmaxf(fmaxf(fabsf(da.x), fabsf(da.y)), fmaxf(fabsf(db.x), fabsf(db.y))));
        const uint32_t lo = __byte_perm(__float_as_uint(ta.x), __float_as_uint(ta.y), 0x5140);
        const uint32_t hi = __byte_perm(__float_as_uint(tb.x), __float_as_uint(tb.y), 0x5140);
        w[k] = fast_row ? __byte_perm(lo, hi, 0x5410) : 0u;
    }
    const bool near = sc > 0.f && (!fast_row || dmax > 0.5f - 0x1p-16f);
    if (__any_sync(0xffffffffu, near) && sc > 0.f) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            w[k] = pack4(__float2int_rn(__fdiv_rn(x[k].x, sc)), __float2int_rn(__fdiv_rn(x[k].y, sc)),
                         __float2int_rn(__fdiv_rn(x[k].z, sc)), __float2int_rn(__fdiv_rn(x[k].w, sc)));
    }
    return sc;
}

// Element k * 4 + u of the quarter goes to byte qq * 32 + k * 4 + u of the row, in the same
// rotated order as the loads.
__device__ __forceinline__ void store_codes(const uint32_t (&w)[8], uint8_t *crow, int qq, int rot) {
#pragma unroll
    for (int k = 0; k < 8; ++k) reinterpret_cast<uint32_t *>(crow)[qq * 8 + ((k + rot) & 7)] = w[k];
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
    volatile int *dvalid = reinterpret_cast<volatile int *>(sm + G::MISC + 64);  // [ND] per destination slot
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + G::MISC + 128);           // [NS] source loaded (tx)
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

    if (warp >= kQtCompute / 32) {
        // ------------------------------------------------------------------ load and store warps
        // Page ids of an item's list live in the warp's registers (lane i: ids i and i + 32);
        // ids from 64 on are read from global memory where needed.
        const bool loader = warp == kQtCompute / 32;
        const PoolView &v = loader ? sv : dv;
        const int32_t *pl = loader ? spl : dpl;
        constexpr int kIds = 2;
        struct Ids { int32_t id[kIds]; };
        auto list_of = [&](int m) {
            return pl + (int64_t)((blockIdx.x + m * gridDim.x) / a.H) * v.pages_per_object;
        };
        auto fetch_ids = [&](int m, Ids &x) {
            const int32_t *l = list_of(m);
#pragma unroll
            for (int u = 0; u < kIds; ++u) {
                const int i = lane + 32 * u;
                x.id[u] = i < v.pages_per_object ? l[i] : 0;
            }
        };
        // The record of head hh, piece by piece (at most one piece per page it touches): the whole
        // warp walks the pieces, the page id comes from the registers, lane 0 issues the copy.
        auto pieces = [&](const Ids &x, const int32_t *list, int hh, uint32_t bytes, auto &&fn) {
            const uint32_t PB = (uint32_t)v.page_bytes;
            uint32_t off = (uint32_t)(hh * v.rec_bytes), at = 0;
            while (at < bytes) {
                const uint32_t pi = qt_page_of(v, off), in = off - pi * PB;
                const uint32_t len = bytes - at < PB - in ? bytes - at : PB - in;
                int32_t id = __shfl_sync(0xffffffffu, pi < 32 ? x.id[0] : x.id[1], pi & 31);
                if (pi >= 64) id = list[pi];
                if (lane == 0) fn(v.base + (uint64_t)id * v.page_bytes + in, at, len);
                off += len;
                at += len;
            }
        };
        Ids cur, nxt, nxt2;   // page ids of items n, n + 1, n + 2
        int n = 0;
        if (blockIdx.x < total) fetch_ids(0, cur);
        if (blockIdx.x + (int)gridDim.x < total) fetch_ids(1, nxt);
        for (;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            // two items ahead, so that the global reads overlap two steps even when the warp runs
            // ahead of the compute warps
            if (item + 2 * (int)gridDim.x < total) fetch_ids(n + 2, nxt2);
            const int32_t *l = list_of(n);
            int stop = 0;
            // every page id of this warp's list in range (ids from 64 on read from the list), or
            // the item is skipped and flagged: the loader does not load it, the store warp does
            // not store it
            bool ok = true;
#pragma unroll
            for (int u = 0; u < kIds; ++u) ok = ok && (uint32_t)cur.id[u] < (uint32_t)v.num_pages;
            for (int i = lane + 32 * kIds; i < v.pages_per_object; i += 32) ok = ok && (uint32_t)l[i] < (uint32_t)v.num_pages;
            ok = __all_sync(0xffffffffu, ok);
            if (loader) {
                // load item n once compute has taken the item that used its source slot
                const int bs = n % NS;
                if (lane == 0 && (*err || (n >= NS && !ptx::mbar_wait(&sfree[bs], (uint32_t)(((n - NS) / NS) & 1), err))))
                    stop = 1;
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
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
                    pieces(cur, l, item % a.H, G::SB, [&](uint8_t *g, uint32_t at, uint32_t len) {
                        ptx::bulk_load(sm + bs * G::SB + at, g, len, &full[bs]);
                    });
            } else {
                // store item n once compute has written it; its slot is free when read out
                const int bd = n % ND;
                if (lane == 0 && !ptx::mbar_wait(&dfull[bd], (uint32_t)((n / ND) & 1), err)) stop = 1;
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
                if (dvalid[bd] && ok)
                    pieces(cur, l, item % a.H, G::DB, [&](uint8_t *g, uint32_t at, uint32_t len) {
                        ptx::bulk_store(g, sm + G::DST0 + bd * G::DB + at, len);
                    });
                else if (!ok && lane == 0)
                    flag_status(a.status, KDA_DEV_BAD_PAGE);
                if (lane == 0) {
                    ptx::bulk_commit();
                    if constexpr (ND == 1) {
                        ptx::bulk_wait_read0();
                        ptx::mbar_arrive(&dfree[bd]);
                    } else {
                        // up to two stores in flight: the older one has read its slot out
                        ptx::bulk_wait_read1();
                        if (n >= 1) ptx::mbar_arrive(&dfree[(n - 1) % ND]);
                    }
                }
            }
            __syncwarp();
            cur = nxt;
            nxt = nxt2;
        }
        if (lane == 0) {
            ptx::bulk_wait0();
            if (loader && *err) {
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
                const bool okw = ptx::mbar_wait(&full[bs], (uint32_t)((n / NS) & 1), err);
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
            if (tid == 0) {
                ptx::mbar_arrive(&sfree[bs]);
                // the destination slot is free once the store of item n - ND has read it out
                const bool okw = n < ND || ptx::mbar_wait(&dfree[bd], (uint32_t)(((n - ND) / ND) & 1), err);
                *go = okw ? 1 : 0;
            }
            if (vld) {
                // codes in registers first; the destination is written once its slot is free
                uint32_t w[8];
                if (QUANT) sc = quant_quarter(x, w);
                tcx::named_bar(1, kQtCompute);
                if (!*go) break;
                if (QUANT) {
                    store_codes(w, dst + 4 * D + r * D, qq, rot);
                    if (qq == 0) reinterpret_cast<float *>(dst)[r] = sc;
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(dst + WQ)[tid] = win;
                } else {
                    dequant_quarter(c8, sc, reinterpret_cast<float *>(dst) + r * D, qq, rot);
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(dst + WF)[tid] = win;
                }
                ptx::fence_proxy_async_smem();
            }
            tcx::named_bar(1, kQtCompute);
            if (tid == 0) {
                dvalid[bd] = vld ? 1 : 0;
                ptx::mbar_arrive(&dfull[bd]);
            }
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
