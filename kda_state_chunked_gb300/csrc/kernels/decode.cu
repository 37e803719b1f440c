// Batched single-token KDA decode step over states gathered through a page table.
//
// Per (request, head): conv of the new token with the stored window (the window shifts by one
// token), then S' = Diag(alpha) S, w = beta (v - S'^T k), S = S' + k w^T, o = S^T q.  The state
// is read from the request's source object and written to its destination object: the same
// object for the in-place step; another one for the ping-pong step, which leaves the source
// object as a checkpoint at the request's position.  The order (decay, delta write, read)
// follows "Lesson 01 · Architecture map", §两种 Attention，两种状态; the fused conv + recurrent
// decode on the state indices follows "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" §0x08
// 8.2.2, the second (ping-pong) slot at a decode checkpoint boundary §0x06 6.7 and 6.8, and the
// block-table gather "Chapitre 8 — Gestion nouvelle génération du cache KV" §8.1 (PagedAttention:
// logical blocks mapped to physical pages through a table).
//
// The step is HBM-bound (about 0.84 flop per byte): every state streams in and out once.
// Two kernels:
//   decode_tma_kernel (bf16, d = 128, pages of at least 64 KiB): one persistent CTA per SM with
//     a three-slot ring of whole records in shared memory; a producer warp bulk-copies the
//     record of a later (request, head) in and the updated record of an earlier one out while
//     sixteen compute warps update the current one, so every SM keeps a record load and a
//     record store in flight.
//   decode_kernel (other shapes): one CTA per (request, head).  Warp w of 16 owns D/16
//     consecutive rows of S; lane l owns D/32 consecutive columns, so every row is one
//     coalesced access of 128-bit loads, the state stays in registers between the two passes,
//     and one shared-memory pass combines the sixteen warps' partial column sums.
#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

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
    const int32_t *dpages = a.dst_pages + (int64_t)b * a.pool.pages_per_object;
    if (tid == 0) {
        ok_s = pages_ok(a.pool, pages) && pages_ok(a.pool, dpages);
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

    // Conv of the new token against the stored window; the shifted window goes to the
    // destination object (the same object for the in-place step).
    const T *qp = static_cast<const T *>(a.q), *kp = static_cast<const T *>(a.k),
            *vp = static_cast<const T *>(a.v);
    for (int c = tid; c < C3; c += kDecThreads) {
        const T *src = c < D ? qp + tok + c : (c < 2 * D ? kp + tok + (c - D) : vp + tok + (c - 2 * D));
        const float x = ld_elem(src);
        const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ((int64_t)h * C3 + c) * 4);
        T pr[kWin];
        float pv[kWin];
#pragma unroll
        for (int u = 0; u < kWin; ++u) {
            pr[u] = *reinterpret_cast<const T *>(obj_addr(a.pool, pages, win_off + ((uint64_t)u * C3 + c) * sizeof(T), a.status));
            pv[u] = ld_elem(&pr[u]);
        }
        xb[c] = w.x * pv[0] + w.y * pv[1] + w.z * pv[2] + w.w * x;
        // every thread has read its window values before any is overwritten (one thread per channel)
        T *wd[kWin];
#pragma unroll
        for (int u = 0; u < kWin; ++u)
            wd[u] = reinterpret_cast<T *>(obj_addr(a.pool, dpages, win_off + ((uint64_t)u * C3 + c) * sizeof(T), a.status));
        *wd[0] = pr[1];
        *wd[1] = pr[2];
        *wd[2] = *src;
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

    // S = S' + k w^T, written to the destination object, and the partial sums of S^T q.
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
        uint8_t *p = obj_addr(a.pool, dpages, rec + ((uint64_t)i * D + lane * VEC) * 4, a.status);
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

// ------------------------------------------------------------------------------------------
// Bulk-copy pipeline for bf16 records of d = 128 (67,840 bytes: S fp32 [128][128], then the
// window [3][384] bf16) in pools of pages of at least 64 KiB.  One persistent CTA per SM walks
// the (request, head) items with a three-slot ring: a producer warp bulk-loads the record of
// item n + 2 (split at page boundaries) and the new token's q, k, v, alpha while sixteen
// compute warps update item n in shared memory; the producer then bulk-stores the updated
// record to its destination.  Every SM thus keeps a record load and a record store in flight.
constexpr int kDtCompute = 512;                  // 16 compute warps
constexpr int kDtThreads = kDtCompute + 32;      // + producer warp
constexpr int kDtSlots = 3;
constexpr uint32_t kDtRec = 67840;               // record bytes (d = 128, bf16)
constexpr uint32_t kDtIn = 1024;                 // q | k | v | alpha of the new token (bf16)
constexpr uint32_t kDtSlot = kDtRec + kDtIn;     // 68,864 (multiple of 128)
constexpr uint32_t DT_RED = kDtSlots * kDtSlot;  // float [4][128] partial column sums
constexpr uint32_t DT_XB = DT_RED + 2048;        // float [384] conv output
constexpr uint32_t DT_MISC = DT_XB + 1536;       // beta per slot, valid flags, barriers
constexpr uint32_t DT_SMEM = DT_MISC + 256;
constexpr int kDtBar = 1;                        // named barrier of the compute warps

__device__ __forceinline__ bool dt_wait(uint64_t *bar, uint32_t parity, volatile int *err) {
    return ptx::mbar_wait(bar, parity, err);
}

__global__ void __launch_bounds__(kDtThreads, 1) decode_tma_kernel(DecodeArgs a) {
    using tcx::named_bar;
    constexpr int D = 128, C3 = 3 * D;
    extern __shared__ __align__(128) uint8_t sm[];
    float *red = reinterpret_cast<float *>(sm + DT_RED);
    float *xb = reinterpret_cast<float *>(sm + DT_XB);
    float *beta_s = reinterpret_cast<float *>(sm + DT_MISC);            // [3]
    volatile int *valid = reinterpret_cast<volatile int *>(sm + DT_MISC + 16);   // [3]
    volatile int *err = reinterpret_cast<volatile int *>(sm + DT_MISC + 32);
    volatile int *go = reinterpret_cast<volatile int *>(sm + DT_MISC + 48);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + DT_MISC + 64);   // [3]
    uint64_t *done = full + kDtSlots;                                   // [3]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.B * a.H;
    const int64_t PB = a.pool.page_bytes;
    if (tid == 0) {
        for (int i = 0; i < kDtSlots; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&done[i], 1);
        }
        *err = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDtCompute / 32) {
        // ------------------------------------------------------------------ producer
        const __nv_bfloat16 *src[4] = {static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
                                      static_cast<const __nv_bfloat16 *>(a.v),
                                      static_cast<const __nv_bfloat16 *>(a.alpha)};
        // walk the record of `item` piece by piece (at most one piece per page it touches)
        auto record_pieces = [&](const int32_t *list, int item, auto &&fn) {
            const int r = item / a.H, hh = item % a.H;
            const int32_t *pages = list + (int64_t)r * a.pool.pages_per_object;
            int64_t off = (int64_t)hh * a.pool.rec_bytes;
            uint32_t done_b = 0;
            while (done_b < kDtRec) {
                const int64_t pi = off / PB, in = off - pi * PB;
                const uint32_t len = (uint32_t)((int64_t)(kDtRec - done_b) < PB - in ? (kDtRec - done_b) : (PB - in));
                fn(pages[pi], in, done_b, len);
                off += len;
                done_b += len;
            }
        };
        auto store_item = [&](int n) {
            const int item = blockIdx.x + n * gridDim.x, b = n % kDtSlots;
            if (!valid[b]) return;
            record_pieces(a.dst_pages, item, [&](int32_t page, int64_t in, uint32_t at, uint32_t len) {
                ptx::bulk_store(a.pool.base + (int64_t)page * PB + in, sm + b * kDtSlot + at, len);
            });
            ptx::bulk_commit();
        };
        // The whole warp walks the items; lane 0 issues the copies and the waits, and all
        // lanes check the request's page ids (a bad id skips the request, as in the other path).
        int n = 0;
        for (;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int b = n % kDtSlots;
            int stop = 0;
            if (lane == 0) {
                if (*err) {
                    stop = 1;
                } else if (n >= kDtSlots) {
                    // the record that used this slot goes back to its pages first
                    if (!dt_wait(&done[b], (uint32_t)(((n - kDtSlots) / kDtSlots) & 1), err)) {
                        stop = 1;
                    } else {
                        store_item(n - kDtSlots);
                        ptx::bulk_wait_read0();
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            const int32_t *pages = a.state_pages + (int64_t)(item / a.H) * a.pool.pages_per_object;
            const int32_t *dpages = a.dst_pages + (int64_t)(item / a.H) * a.pool.pages_per_object;
            bool ok = true;
            for (int i = lane; i < a.pool.pages_per_object; i += 32)
                ok = ok && (uint32_t)pages[i] < (uint32_t)a.pool.num_pages && (uint32_t)dpages[i] < (uint32_t)a.pool.num_pages;
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                valid[b] = ok ? 1 : 0;
                if (!ok) {
                    flag_status(a.status, KDA_DEV_BAD_PAGE);
                    ptx::mbar_arrive(&full[b]);
                } else {
                    ptx::mbar_arrive_expect_tx(&full[b], kDtSlot);
                    record_pieces(a.state_pages, item, [&](int32_t page, int64_t in, uint32_t at, uint32_t len) {
                        ptx::bulk_load(sm + b * kDtSlot + at, a.pool.base + (int64_t)page * PB + in, len, &full[b]);
                    });
                    const int64_t tok = (int64_t)item * D;   // [B][H][D] with item = r * H + h
                    for (int x = 0; x < 4; ++x)
                        ptx::bulk_load(sm + b * kDtSlot + kDtRec + x * 256, src[x] + tok, 256, &full[b]);
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            // the last records (every slot still holding one) go back too
            for (int m = n - kDtSlots < 0 ? 0 : n - kDtSlots; m < n && !*err; ++m) {
                const int b = m % kDtSlots;
                if (!dt_wait(&done[b], (uint32_t)((m / kDtSlots) & 1), err)) break;
                store_item(m);
            }
            ptx::bulk_wait0();
            if (*err) {
                // leave no copy in flight
                for (int m = n - kDtSlots < 0 ? 0 : n - kDtSlots; m < n; ++m) {
                    uint32_t k = 0;
                    while (!ptx::mbar_try_wait(&full[m % kDtSlots], (uint32_t)((m / kDtSlots) & 1)) && k < ptx::kSpinLimit) ++k;
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ compute
        const int j = tid & (D - 1), rq = tid >> 7;          // value channel, row quarter
        for (int n = 0;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int b = n % kDtSlots, hh = item % a.H;
            // thread 0 waits for the slot and decides for all compute threads whether to go on
            if (tid == 0) *go = (dt_wait(&full[b], (uint32_t)((n / kDtSlots) & 1), err) && !*err) ? 1 : 0;
            named_bar(kDtBar, kDtCompute);
            if (!*go) break;
            uint8_t *slot = sm + b * kDtSlot;
            float *S = reinterpret_cast<float *>(slot);
            __nv_bfloat16 *win = reinterpret_cast<__nv_bfloat16 *>(slot + D * D * 4);
            const __nv_bfloat16 *xin = reinterpret_cast<const __nv_bfloat16 *>(slot + kDtRec);
            if (valid[b]) {
                // conv of the new token with the window; the window shifts in the slot
                if (tid < C3) {
                    const int c = tid;
                    const float x = __bfloat162float(xin[c]);
                    const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ((int64_t)hh * C3 + c) * 4);
                    const __nv_bfloat16 p0 = win[c], p1 = win[C3 + c], p2 = win[2 * C3 + c];
                    xb[c] = w.x * __bfloat162float(p0) + w.y * __bfloat162float(p1) + w.z * __bfloat162float(p2) + w.w * x;
                    win[c] = p1;
                    win[C3 + c] = p2;
                    win[2 * C3 + c] = xin[c];
                }
                if (tid == 0) beta_s[b] = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.beta)[item]);
                named_bar(kDtBar, kDtCompute);
                // S' = Diag(alpha) S; partial column sums of S'^T k over this thread's 32 rows
                float sv[32];
                float acc = 0.f;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = rq * 32 + ii;
                    sv[ii] = __bfloat162float(xin[3 * D + i]) * S[i * D + j];
                    acc = fmaf(xb[D + i], sv[ii], acc);
                }
                red[rq * D + j] = acc;
                named_bar(kDtBar, kDtCompute);
                const float u = (red[j] + red[D + j]) + (red[2 * D + j] + red[3 * D + j]);
                const float wj = beta_s[b] * (xb[2 * D + j] - u);
                named_bar(kDtBar, kDtCompute);   // red is reused below
                // S = S' + k w^T in the slot, and the partial sums of S^T q
                float ao = 0.f;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = rq * 32 + ii;
                    const float v = fmaf(xb[D + i], wj, sv[ii]);
                    S[i * D + j] = v;
                    ao = fmaf(xb[i], v, ao);
                }
                red[rq * D + j] = ao;
                ptx::fence_proxy_async_smem();
                named_bar(kDtBar, kDtCompute);
                if (rq == 0) {
                    const float o = (red[j] + red[D + j]) + (red[2 * D + j] + red[3 * D + j]);
                    static_cast<__nv_bfloat16 *>(a.o)[(int64_t)item * D + j] = __float2bfloat16_rn(o);
                }
            }
            // the slot may be stored (and, once the store has read it, refilled); red and xb
            // are free for the next item
            named_bar(kDtBar, kDtCompute);
            if (tid == 0) ptx::mbar_arrive(&done[b]);
        }
    }
    __syncthreads();
    if (*err && tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
}


// ------------------------------------------------------------------------------------------
// Fused speculative verify for bf16 records of d = 128 in pools of pages of at least 64 KiB:
// K draft tokens per (request, head) applied one after another ("KIMI K3 경량 복제에서 본 KDA의
// AI 인프라 과제", §0x06 6.4: the verify pass keeps the intermediate states).  One persistent
// CTA per SM walks the (request, head) items.  The producer warp bulk-loads an item's source
// record and its K draft tokens once; the sixteen compute warps move S into registers (thread
// = one value column and 32 key rows) and the window and drafts into a token history, which
// frees the input buffer for the next item's load.  For every draft token they run the same
// step as decode (conv, S' = Diag(alpha) S, w = beta (v - S'^T k), S = S' + k w^T, o = S^T q)
// and write the resulting record (S and the window after that token) into one of two output
// buffers; compute thread 0 bulk-stores it into that token's object right away, so two
// record stores can be in flight while the next draft runs.  The source object is only read.
// Traffic per item: one record read and K record writes.
constexpr int kVfMaxK = kVerifyFusedMaxK;
constexpr uint32_t VF_IN = 0;                                  // record, then inputs [K][q|k|v|alpha]
constexpr uint32_t VF_INPUTS = kDtRec;                         // 1 KiB per draft token
constexpr uint32_t VF_OUT = kDtRec + kVfMaxK * kDtIn;          // two output records
constexpr uint32_t VF_HIST = VF_OUT + 2 * kDtRec;              // bf16 window [3][384], drafts [K][512]
constexpr uint32_t VF_HIST_DRAFT = VF_HIST + 3 * 768;
constexpr uint32_t VF_RED = VF_HIST_DRAFT + kVfMaxK * 1024;    // float [4][128]
constexpr uint32_t VF_XB = VF_RED + 2048;                      // float [384]
constexpr uint32_t VF_MISC = VF_XB + 1536;                     // betas, flags, barriers
constexpr uint32_t VF_SMEM = VF_MISC + 256;
static_assert(VF_OUT % 128 == 0 && VF_HIST % 16 == 0 && VF_SMEM <= 227 * 1024, "verify shared memory layout");

__global__ void __launch_bounds__(kDtThreads, 1) verify_tma_kernel(VerifyArgs a) {
    using tcx::named_bar;
    constexpr int D = 128, C3 = 3 * D;
    extern __shared__ __align__(128) uint8_t sm[];
    float *red = reinterpret_cast<float *>(sm + VF_RED);
    float *xb = reinterpret_cast<float *>(sm + VF_XB);
    float *beta_s = reinterpret_cast<float *>(sm + VF_MISC);                 // [K]
    volatile int *valid = reinterpret_cast<volatile int *>(sm + VF_MISC + 32);
    volatile int *err = reinterpret_cast<volatile int *>(sm + VF_MISC + 36);
    volatile int *go = reinterpret_cast<volatile int *>(sm + VF_MISC + 40);
    uint64_t *in_full = reinterpret_cast<uint64_t *>(sm + VF_MISC + 48);
    uint64_t *in_free = in_full + 1;
    const __nv_bfloat16 *hist_win = reinterpret_cast<const __nv_bfloat16 *>(sm + VF_HIST);
    const __nv_bfloat16 *hist_draft = reinterpret_cast<const __nv_bfloat16 *>(sm + VF_HIST_DRAFT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.B * a.H, K = a.K;
    const int64_t PB = a.pool.page_bytes;
    const int P = a.pool.pages_per_object;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) ptx::mbar_init(&in_full[i], 1);
        *err = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDtCompute / 32) {
        // ------------------------------------------------------------------ producer
        const __nv_bfloat16 *src[4] = {static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
                                      static_cast<const __nv_bfloat16 *>(a.v),
                                      static_cast<const __nv_bfloat16 *>(a.alpha)};
        // the record of head hh in the object whose page list is `pages`, piece by piece
        // (at most one piece per page it touches)
        auto record_pieces = [&](const int32_t *pages, int hh, auto &&fn) {
            int64_t off = (int64_t)hh * a.pool.rec_bytes;
            uint32_t done_b = 0;
            while (done_b < kDtRec) {
                const int64_t pi = off / PB, in = off - pi * PB;
                const uint32_t len = (uint32_t)((int64_t)(kDtRec - done_b) < PB - in ? (kDtRec - done_b) : (PB - in));
                fn(pages[pi], in, done_b, len);
                off += len;
                done_b += len;
            }
        };
        // check the request's page ids (source and every draft object; the whole warp) and,
        // when they are valid, load the item's record and draft tokens (lane 0)
        auto issue_load = [&](int n) -> bool {
            const int item = blockIdx.x + n * gridDim.x, r = item / a.H;
            const int32_t *sp = a.src_pages + (int64_t)r * P;
            bool ok = true;
            for (int i = lane; i < P; i += 32) ok = ok && (uint32_t)sp[i] < (uint32_t)a.pool.num_pages;
            for (int jd = 0; jd < K; ++jd) {
                const int32_t *ip = a.inter_pages + ((int64_t)jd * a.B + r) * P;
                for (int i = lane; i < P; i += 32) ok = ok && (uint32_t)ip[i] < (uint32_t)a.pool.num_pages;
            }
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                *valid = ok ? 1 : 0;
                if (!ok) {
                    flag_status(a.status, KDA_DEV_BAD_PAGE);
                    ptx::mbar_arrive(in_full);
                } else {
                    ptx::mbar_arrive_expect_tx(in_full, kDtRec + (uint32_t)K * kDtIn);
                    record_pieces(sp, item % a.H, [&](int32_t page, int64_t in, uint32_t at, uint32_t len) {
                        ptx::bulk_load(sm + VF_IN + at, a.pool.base + (int64_t)page * PB + in, len, in_full);
                    });
                    for (int jd = 0; jd < K; ++jd) {
                        const int64_t tok = ((int64_t)jd * total + item) * D;
                        for (int x = 0; x < 4; ++x)
                            ptx::bulk_load(sm + VF_INPUTS + jd * kDtIn + x * 256, src[x] + tok, 256, in_full);
                    }
                }
            }
            __syncwarp();
            return ok;
        };
        int issued = 0;
        if (blockIdx.x < total) {
            (void)issue_load(0);
            issued = 1;
        }
        for (int n = 0;; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            int stop = 0;
            // the compute warps have taken item n out of the input buffer
            if (lane == 0 && (*err || !dt_wait(in_free, (uint32_t)(n & 1), err))) stop = 1;
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            if (item + (int)gridDim.x < total) {
                (void)issue_load(n + 1);
                issued = n + 2;
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (*err && issued > 0) {
                // leave no load in flight: only the last issued one can be pending
                uint32_t k = 0;
                while (!ptx::mbar_try_wait(in_full, (uint32_t)((issued - 1) & 1)) && k < ptx::kSpinLimit) ++k;
            }
        }
    } else {
        // ------------------------------------------------------------------ compute
        const int j = tid & (D - 1), rq = tid >> 7;          // value channel, row quarter
        // *go is written by thread 0 before a barrier and read by every thread right after it;
        // the next write comes after at least one more barrier, so all threads agree on it
        int gv = 0;
        bool alive = true;
        for (int n = 0; alive; ++n) {
            const int item = blockIdx.x + n * gridDim.x;
            if (item >= total) break;
            const int hh = item % a.H;
            if (tid == 0) *go = (dt_wait(in_full, (uint32_t)(n & 1), err) && !*err) ? 1 : 0;
            named_bar(kDtBar, kDtCompute);
            alive = *go != 0;
            if (!alive) break;
            const bool ok = *valid != 0;
            float sv[32];
            if (ok) {
                const float *S = reinterpret_cast<const float *>(sm + VF_IN);
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) sv[ii] = S[(rq * 32 + ii) * D + j];
                // window rows and draft tokens into the history (16 bytes per thread and step)
                const uint4 *win = reinterpret_cast<const uint4 *>(sm + VF_IN + D * D * 4);
                for (int x = tid; x < 3 * C3 * 2 / 16; x += kDtCompute)
                    reinterpret_cast<uint4 *>(sm + VF_HIST)[x] = win[x];
                for (int x = tid; x < K * (int)kDtIn / 16; x += kDtCompute)
                    reinterpret_cast<uint4 *>(sm + VF_HIST_DRAFT)[x] = reinterpret_cast<const uint4 *>(sm + VF_INPUTS)[x];
                if (tid < K) beta_s[tid] = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.beta)[(int64_t)tid * total + item]);
            }
            named_bar(kDtBar, kDtCompute);
            if (tid == 0) ptx::mbar_arrive(in_free);   // the input buffer may take the next item
            if (!ok) continue;
            // raw token r of the sequence window | drafts: r < 3 from the window, else draft r - 3
            auto raw = [&](int r, int c) -> float {
                return __bfloat162float(r < 3 ? hist_win[r * C3 + c] : hist_draft[(r - 3) * 512 + c]);
            };
            for (int jd = 0; jd < K; ++jd, ++gv) {
                const int ob = gv & 1;
                if (tid < C3) {
                    const int c = tid;
                    const float4 w = *reinterpret_cast<const float4 *>(a.conv_w + ((int64_t)hh * C3 + c) * 4);
                    xb[c] = w.x * raw(jd, c) + w.y * raw(jd + 1, c) + w.z * raw(jd + 2, c) + w.w * raw(jd + 3, c);
                }
                // the output buffer's previous record has been read by its bulk store (thread 0
                // issued both stores since: at most the newer one may still be reading)
                if (tid == 0 && gv >= 2) ptx::bulk_wait_read1();
                named_bar(kDtBar, kDtCompute);
                // S' = Diag(alpha) S; partial column sums of S'^T k over this thread's 32 rows
                float acc = 0.f;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = rq * 32 + ii;
                    sv[ii] *= __bfloat162float(hist_draft[jd * 512 + C3 + i]);
                    acc = fmaf(xb[D + i], sv[ii], acc);
                }
                red[rq * D + j] = acc;
                named_bar(kDtBar, kDtCompute);
                const float u = (red[j] + red[D + j]) + (red[2 * D + j] + red[3 * D + j]);
                const float wj = beta_s[jd] * (xb[2 * D + j] - u);
                named_bar(kDtBar, kDtCompute);   // red is reused below
                // S = S' + k w^T into the output record, and the partial sums of S^T q
                float *So = reinterpret_cast<float *>(sm + VF_OUT + ob * kDtRec);
                float ao = 0.f;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = rq * 32 + ii;
                    sv[ii] = fmaf(xb[D + i], wj, sv[ii]);
                    So[i * D + j] = sv[ii];
                    ao = fmaf(xb[i], sv[ii], ao);
                }
                red[rq * D + j] = ao;
                // the window after this token: raw tokens jd + 1 .. jd + 3
                if (tid < 3 * C3 / 8) {
                    const int u = tid / (C3 / 8), c = (tid % (C3 / 8)) * 8, r = jd + 1 + u;
                    const uint4 v4 = r < 3 ? *reinterpret_cast<const uint4 *>(hist_win + r * C3 + c)
                                           : *reinterpret_cast<const uint4 *>(hist_draft + (r - 3) * 512 + c);
                    *reinterpret_cast<uint4 *>(sm + VF_OUT + ob * kDtRec + D * D * 4 + (u * C3 + c) * 2) = v4;
                }
                ptx::fence_proxy_async_smem();
                named_bar(kDtBar, kDtCompute);
                if (tid == 0) {
                    // the record after draft jd into its object, piece by piece (at most one piece
                    // per page it touches), from the buffer just written
                    const int32_t *ip = a.inter_pages + ((int64_t)jd * a.B + item / a.H) * P;
                    int64_t off = (int64_t)hh * a.pool.rec_bytes;
                    uint32_t at = 0;
                    while (at < kDtRec) {
                        const int64_t pi = off / PB, in = off - pi * PB;
                        const uint32_t len = (uint32_t)((int64_t)(kDtRec - at) < PB - in ? (kDtRec - at) : (PB - in));
                        ptx::bulk_store(a.pool.base + (int64_t)ip[pi] * PB + in, sm + VF_OUT + ob * kDtRec + at, len);
                        off += len;
                        at += len;
                    }
                    ptx::bulk_commit();
                }
                if (rq == 0) {
                    const float o = (red[j] + red[D + j]) + (red[2 * D + j] + red[3 * D + j]);
                    static_cast<__nv_bfloat16 *>(a.o)[((int64_t)jd * total + item) * D + j] = __float2bfloat16_rn(o);
                }
                named_bar(kDtBar, kDtCompute);   // red and xb are reused by the next token
            }
        }
        if (tid == 0) ptx::bulk_wait_read0();   // the last records have left their buffers
    }
    __syncthreads();
    if (*err && tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (a.d == 128 && a.dtype == KDA_BF16 && a.pool.rec_bytes == (int64_t)kDtRec && a.pool.page_bytes >= 65536) {
        int dev = 0, nsm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DT_SMEM);
        if (e != cudaSuccess) return e;
        const int total = a.B * a.H;
        decode_tma_kernel<<<(unsigned)(total < nsm ? total : nsm), kDtThreads, DT_SMEM, s>>>(a);
        return cudaGetLastError();
    }
    if (a.d == 128) return a.dtype == KDA_BF16 ? launch_decode_t<128, __nv_bfloat16>(a, s)
                                               : launch_decode_t<128, float>(a, s);
    if (a.d == 64) return a.dtype == KDA_BF16 ? launch_decode_t<64, __nv_bfloat16>(a, s)
                                              : launch_decode_t<64, float>(a, s);
    return cudaErrorInvalidValue;
}

bool verify_fused_supported(const VerifyArgs &a) {
    return a.d == 128 && a.dtype == KDA_BF16 && a.pool.rec_bytes == (int64_t)kDtRec && a.pool.page_bytes >= 65536 &&
           a.K >= 1 && a.K <= kVfMaxK;
}

cudaError_t launch_verify_fused(const VerifyArgs &a, cudaStream_t s) {
    if (a.B <= 0) return cudaSuccess;
    if (!verify_fused_supported(a)) return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)VF_SMEM);
    if (e != cudaSuccess) return e;
    const int total = a.B * a.H;
    verify_tma_kernel<<<(unsigned)(total < nsm ? total : nsm), kDtThreads, VF_SMEM, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
