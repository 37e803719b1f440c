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
// pages of at least 4 KiB.  One persistent CTA per SM walks the head records with a ring of
// three record slots: a producer warp bulk-loads a record (split at page boundaries) into one
// slot and bulk-stores the converted record of the item three back, while sixteen compute
// warps convert another slot in place: every thread first reads its part of the source record
// into registers, then, after a barrier, writes its part of the converted record over it
// (warp w: rows w, w + 16, ...; a lane takes 4 consecutive values of a row, the row's max-abs
// is a warp reduction).  The codes are those of the kernels above, bit for bit: the division
// goes through the reciprocal where that provably gives the same integer (see below), through
// the IEEE division elsewhere.  Page ids of an item are checked before the producer waits for its slot, so that the
// check's global reads are off the pipeline's critical path.
constexpr int kQtCompute = 512;
constexpr int kQtThreads = kQtCompute + 32;
constexpr int kQtSlots = 3;
constexpr uint32_t kQtFull = 67840, kQtQ8 = 19200;
constexpr uint32_t kQtSlot = kQtFull;             // a slot holds the larger of the two records
constexpr uint32_t QT_MISC = kQtSlots * kQtSlot;
constexpr uint32_t QT_SMEM = QT_MISC + 256;
static_assert(kQtSlot % 128 == 0 && QT_SMEM <= 227 * 1024, "INT8 pipeline shared memory");

// Page index of in-object byte offset `off` (below 4 GiB): a shift for power-of-two page
// sizes, otherwise the high half of off * ceil(2^32 / page_bytes) corrected by one compare.
__device__ __forceinline__ uint32_t qt_page_of(const PoolView &v, uint32_t off) {
    if (v.page_shift >= 0) return off >> v.page_shift;
    uint32_t q = __umulhi(off, v.page_magic);
    if ((uint64_t)q * (uint64_t)v.page_bytes > off) --q;
    return q;
}

template <bool QUANT>
__global__ void __launch_bounds__(kQtThreads, 1) q8_tma_kernel(Q8Args a) {
    constexpr int D = 128;
    constexpr int RPW = D / (kQtCompute / 32);   // rows per compute warp (8)
    extern __shared__ __align__(128) uint8_t sm[];
    volatile int *valid = reinterpret_cast<volatile int *>(sm + QT_MISC);        // [3]
    volatile int *err = reinterpret_cast<volatile int *>(sm + QT_MISC + 16);
    volatile int *go = reinterpret_cast<volatile int *>(sm + QT_MISC + 20);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + QT_MISC + 32);            // [3]
    uint64_t *done = full + kQtSlots;                                            // [3]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.n * a.H;
    // source and destination side of this direction
    const PoolView &sv = QUANT ? a.full : a.q8, &dv = QUANT ? a.q8 : a.full;
    const int32_t *spl = QUANT ? a.full_pages : a.q8_pages, *dpl = QUANT ? a.q8_pages : a.full_pages;
    const uint32_t s_bytes = QUANT ? kQtFull : kQtQ8, d_bytes = QUANT ? kQtQ8 : kQtFull;
    if (tid == 0) {
        for (int i = 0; i < 2 * kQtSlots; ++i) ptx::mbar_init(&full[i], 1);
        *err = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kQtCompute / 32) {
        // ------------------------------------------------------------------ producer
        // record of head hh of the object with page list `pages` in view `v`, piece by piece
        auto pieces = [&](const PoolView &v, const int32_t *pages, int hh, uint32_t bytes, auto &&fn) {
            const uint32_t PB = (uint32_t)v.page_bytes;
            uint32_t off = (uint32_t)(hh * v.rec_bytes), at = 0;
            while (at < bytes) {
                const uint32_t pi = qt_page_of(v, off), in = off - pi * PB;
                const uint32_t len = bytes - at < PB - in ? bytes - at : PB - in;
                fn(v.base + (uint64_t)pages[pi] * v.page_bytes + in, at, len);
                off += len;
                at += len;
            }
        };
        auto store_item = [&](int m) {
            const int item = blockIdx.x + m * gridDim.x, b = m % kQtSlots;
            if (!valid[b]) return;
            pieces(dv, dpl + (int64_t)(item / a.H) * dv.pages_per_object, item % a.H, d_bytes,
                   [&](uint8_t *g, uint32_t at, uint32_t len) { ptx::bulk_store(g, sm + b * kQtSlot + at, len); });
            ptx::bulk_commit();
        };
        int n = 0;
        for (;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int b = n % kQtSlots;
            // page ids of this item first (the whole warp), then the slot
            const int obj = item / a.H;
            const int32_t *sp = spl + (int64_t)obj * sv.pages_per_object, *dp = dpl + (int64_t)obj * dv.pages_per_object;
            bool ok = true;
            for (int i = lane; i < sv.pages_per_object; i += 32) ok = ok && (uint32_t)sp[i] < (uint32_t)sv.num_pages;
            for (int i = lane; i < dv.pages_per_object; i += 32) ok = ok && (uint32_t)dp[i] < (uint32_t)dv.num_pages;
            ok = __all_sync(0xffffffffu, ok);
            int stop = 0;
            if (lane == 0) {
                if (*err) {
                    stop = 1;
                } else if (n >= kQtSlots) {
                    // the item that used this slot goes out first
                    if (!ptx::mbar_wait(&done[b], (uint32_t)(((n - kQtSlots) / kQtSlots) & 1), err)) {
                        stop = 1;
                    } else {
                        store_item(n - kQtSlots);
                        ptx::bulk_wait_read0();
                    }
                }
                if (!stop) {
                    valid[b] = ok ? 1 : 0;
                    if (!ok) {
                        flag_status(a.status, KDA_DEV_BAD_PAGE);
                        ptx::mbar_arrive(&full[b]);
                    } else {
                        ptx::mbar_arrive_expect_tx(&full[b], s_bytes);
                        pieces(sv, sp, item % a.H, s_bytes, [&](uint8_t *g, uint32_t at, uint32_t len) {
                            ptx::bulk_load(sm + b * kQtSlot + at, g, len, &full[b]);
                        });
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        if (lane == 0) {
            for (int m = n - kQtSlots < 0 ? 0 : n - kQtSlots; m < n && !*err; ++m) {
                if (!ptx::mbar_wait(&done[m % kQtSlots], (uint32_t)((m / kQtSlots) & 1), err)) break;
                store_item(m);
            }
            ptx::bulk_wait0();
            if (*err) {
                // leave no load in flight
                for (int m = n - kQtSlots < 0 ? 0 : n - kQtSlots; m < n; ++m) {
                    uint32_t k = 0;
                    while (!ptx::mbar_try_wait(&full[m % kQtSlots], (uint32_t)((m / kQtSlots) & 1)) && k < ptx::kSpinLimit) ++k;
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ compute
        // full record: S fp32 at 0, window at D*D*4; INT8 record: scales at 0, codes at 4 D,
        // window at 4 D + D*D
        constexpr uint32_t WF = D * D * 4, WQ = 4 * D + D * D, WBYTES = 9 * D * 2;
        for (int n = 0;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int b = n % kQtSlots;
            if (tid == 0) *go = (ptx::mbar_wait(&full[b], (uint32_t)((n / kQtSlots) & 1), err) && !*err) ? 1 : 0;
            tcx::named_bar(1, kQtCompute);
            if (!*go) break;
            if (valid[b]) {
                uint8_t *slot = sm + b * kQtSlot;
                float *S = reinterpret_cast<float *>(slot);
                float *scale = reinterpret_cast<float *>(slot);
                uint32_t *codes = reinterpret_cast<uint32_t *>(slot + 4 * D);
                uint4 w = make_uint4(0, 0, 0, 0);
                if (QUANT) {
                    float4 x[RPW];
#pragma unroll
                    for (int k = 0; k < RPW; ++k) x[k] = reinterpret_cast<const float4 *>(S + (warp + 16 * k) * D)[lane];
                    if (tid < WBYTES / 16) w = reinterpret_cast<const uint4 *>(slot + WF)[tid];
                    tcx::named_bar(1, kQtCompute);   // the whole source record is in registers
#pragma unroll
                    for (int k = 0; k < RPW; ++k) {
                        const int r = warp + 16 * k;
                        float m = fmaxf(fmaxf(fabsf(x[k].x), fabsf(x[k].y)), fmaxf(fabsf(x[k].z), fabsf(x[k].w)));
                        m = warp_max(m);
                        const float sc = __fdiv_rn(m, 127.f);
                        const float xs[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
                        // code = rint(RN(x / sc)) through the correctly rounded reciprocal, with
                        // Ziv's rounding test: y = RN(x RN(1/sc)) lies within 127 * 2^-23 +
                        // 2^-18 < 2^-14 of RN(x / sc) (|x / sc| <= 127), so rint(y) is that
                        // integer unless y is within 2^-14 of a half-integer.  Such elements,
                        // and rows whose reciprocal is not finite, take the IEEE division; the
                        // branch is taken per warp and only when a lane needs it.
                        const float rs = __frcp_rn(sc);
                        const bool fast_row = sc > 0.f && isfinite(rs);
                        int qv[4];
                        bool near = !fast_row && sc > 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float y = __fmul_rn(xs[u], rs), ay = fabsf(y);
                            near = near || fabsf(ay - floorf(ay) - 0.5f) < 0x1p-14f;
                            qv[u] = fast_row ? __float2int_rn(y) : 0;
                        }
                        if (__any_sync(0xffffffffu, near)) {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                if (sc > 0.f) qv[u] = __float2int_rn(__fdiv_rn(xs[u], sc));
                        }
                        uint32_t packed = 0;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int q = qv[u] > 127 ? 127 : (qv[u] < -127 ? -127 : qv[u]);
                            packed |= (uint32_t)(q & 0xff) << (8 * u);
                        }
                        codes[r * (D / 4) + lane] = packed;
                        if (lane == 0) scale[r] = sc;
                    }
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(slot + WQ)[tid] = w;
                } else {
                    uint32_t c[RPW];
                    float sc[RPW];
#pragma unroll
                    for (int k = 0; k < RPW; ++k) {
                        c[k] = codes[(warp + 16 * k) * (D / 4) + lane];
                        sc[k] = scale[warp + 16 * k];
                    }
                    if (tid < WBYTES / 16) w = reinterpret_cast<const uint4 *>(slot + WQ)[tid];
                    tcx::named_bar(1, kQtCompute);   // the whole INT8 record is in registers
#pragma unroll
                    for (int k = 0; k < RPW; ++k) {
                        float4 v;
                        v.x = (float)(signed char)(c[k] & 0xff) * sc[k];
                        v.y = (float)(signed char)((c[k] >> 8) & 0xff) * sc[k];
                        v.z = (float)(signed char)((c[k] >> 16) & 0xff) * sc[k];
                        v.w = (float)(signed char)(c[k] >> 24) * sc[k];
                        reinterpret_cast<float4 *>(S + (warp + 16 * k) * D)[lane] = v;
                    }
                    if (tid < WBYTES / 16) reinterpret_cast<uint4 *>(slot + WF)[tid] = w;
                }
                ptx::fence_proxy_async_smem();
            }
            tcx::named_bar(1, kQtCompute);
            if (tid == 0) ptx::mbar_arrive(&done[b]);
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(q8_tma_kernel<QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QT_SMEM);
    if (e != cudaSuccess) return e;
    const int total = a.n * a.H;
    q8_tma_kernel<QUANT><<<(unsigned)(total < nsm ? total : nsm), kQtThreads, QT_SMEM, s>>>(a);
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
