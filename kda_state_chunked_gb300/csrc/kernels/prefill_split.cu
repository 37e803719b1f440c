// Split chunked prefill on the 5th-generation tensor cores (bf16 inputs, d = 128).
//
// It computes the same result as the fused kernel: the token recurrence
// S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T, o_t = S_t^T q_t after the width-4
// causal conv on q | k | v ("Lesson 01 · Architecture map", §两种 Attention，两种状态), grouped
// into chunks of 64 tokens that each act on S as one affine map ("KIMI K3 경량 복제에서 본 KDA의
// AI 인프라 과제", §0x01 1.3), with checkpoints of (S, conv window) written at listed chunk ends
// ("Cache de préfixe hybride KDA–MLA", §Le fonctionnement du prefill).
//
// Everything of a chunk that does not depend on the state runs in parallel over all
// (chunk, head) items; only the state contractions remain sequential per chain:
//
//   chunk_prep_kernel (one CTA per (item, head), 160 threads, three CTAs per SM)
//     conv, decay factors, Kt' = k gamma_r/gamma_C, Qt' = q gamma_r/gamma_C, Kb = k gamma_C/gamma_r,
//     G | P = [Kt'; Qt'] Kb^T (tcgen05), T = (I + Diag(beta) strict_lower(G))^{-1} Diag(beta)
//     (16 x 16 diagonal inverses on CUDA cores, the rest in three tcgen05 stages),
//     WK'^T = Kt'^T T^T (tcgen05), and writes one operand image
//     per item, bf16 and 128-byte swizzled as the chain kernel's MMAs read it:
//     Gamma_C [-WK' | Qt'] = [-WK' Gamma_C | q gamma_r], Kb, P, V, T, and gamma_C (fp32).  Conv
//     windows of checkpoints are written here.
//
//   chain_kernel (one CTA per (sequence, head), 512 threads)
//     S^T resident in TMEM; per chunk: U^T = V^T T^T, then [W^T | O^T] = [U^T | 0] +
//     S^T (Gamma_C [-WK' | Qt'])^T in one MMA group (the decay is in the image, so the state
//     operand is S itself), S^T <- Gamma_C S^T + W^T Kb,
//     O^T += W^T P^T; checkpoint states and outputs.  Images arrive by bulk copies,
//     double-buffered.
//
// The chunks of every chain are processed in waves; a wave's images use one of two slots.
// All launches go to one stream, each a programmatic dependent launch of the one before:
// prep 0, chains 0, prep 1, chains 1, ...  Chains w are placed once every CTA of prep w has
// started and wait in hardware for prep w to complete (and so for chains w - 1, which hand
// the state on through a small fp32 scratch) before reading anything; each chain CTA then
// allows prep w + 1, so the chains hold their SMs before prep w + 1 fills the rest and the
// two overlap.  Prep w + 1 overwrites the slot chains w - 1 read, which are complete by
// then; its last CTA waits for chains w to complete before it exits.  Every wait of the kernels' own is bounded: on a timeout a kernel
// records KDA_DEV_TIMEOUT, stops issuing work, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "sm100_ptx.cuh"
#include "tc_common.cuh"

namespace kda {

int encode_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows);

namespace {

using namespace tcx;

constexpr int D = 128;
constexpr int C = kChunk;   // 64

// Operand image of one (chunk, head) item (byte offsets; every operand 1024-byte aligned).
constexpr uint32_t IMG_WQ = 0;       // [2 kb][128 rows: -WK' Gamma_C 0-63 | q gamma_r 64-127][128 B]  K-major B
constexpr uint32_t IMG_PK = 32768;   // [3 N blocks: P^T | Kb keys 0-63 | Kb keys 64-127][64 rows j][128 B]  MN-major B
constexpr uint32_t IMG_V = 57344;    // V     [2 kb][64 rows][128 B]   MN-major A operand
constexpr uint32_t IMG_T = 73728;    // T     [64 rows][128 B]         K-major B operand
constexpr uint32_t IMG_GC = 81920;   // gamma_C fp32 [128]
static_assert(IMG_GC + 512 == kImageBytes, "image layout");

__device__ __forceinline__ uint8_t *image_addr(const SplitArgs &a, int wave, int64_t idx_in_wave, int h) {
    const int64_t slot = wave & 1;
    return a.images + ((slot * a.slot_items + idx_in_wave) * a.p.H + h) * kImageBytes;
}

// ============================================================================ chunk prep
constexpr int kAThreads = 160;   // warps 0-3 compute, warp 4 TMA + MMA + bulk stores

// Shared memory (73 KiB: three CTAs per SM).
constexpr uint32_t A_KQ = 0;        // [2 kb][128 rows: k 0-63 | q 64-127][128 B] -> Kt' | Qt'
constexpr uint32_t A_T = 8192;      // T [64][128 B], over the first Qt' half once M1 has read it
constexpr uint32_t A_V = 32768;     // [2 kb][64][128 B]  raw v (V goes to the image) -> solve tiles
constexpr uint32_t A_AL = 49152;    // [2 kb][64][128 B]  raw alpha -> Kb -> fp32 solve scratch
constexpr uint32_t A_DG = 65536;    // float [64][16]     partial sums of the diagonal q.k
constexpr uint32_t A_GC = 69632;    // float [128]  gamma_C
constexpr uint32_t A_BS = 70144;    // float [64]   beta
constexpr uint32_t A_PD = 70400;    // float [64]   exact diagonal of P
constexpr uint32_t A_RED = 70656;   // float2 [2][64] half products of alpha
constexpr uint32_t A_HALO = 71680;  // bf16 [3][384] conv window
constexpr uint32_t A_BAR = 73984;   // mbarriers, flags
constexpr uint32_t A_SMEM = A_BAR + 128 + 1024;
// three CTAs per SM: 228 KiB of shared memory per SM, 1 KiB of it reserved per CTA
static_assert(3 * (A_SMEM + 1024) <= 228 * 1024, "three chunk-prep CTAs per SM");
constexpr int kAWg = 1, kAHalf = 2;   // named barriers (128 and 64 threads)

enum { AB_FULL = 0, AB_P1, AB_GP, AB_KBF, AB_T, AB_M2, AB_SO, A_NBARS };
// bf16 64 x 64 tiles of the tensor-core solve (8 KiB each, row-major, 128-byte swizzle).  The A
// operand of an M = 128 product reads its rows 64-127 8 KiB after rows 0-63, and each A tile has
// a copy there, so TMEM lanes 64-127 hold the product's rows 0-63 once more and all four compute
// warps share an epilogue, each thread half a row.  Binv over the second Qt' half (read by M1),
// its copy over the first raw v half; N over the second raw v half; E, then E^2, over the raw v
// tile with its copy in the second half (each once the previous stage has read that tile); G
// over Binv once stage 2 has read it; T at A_T.
constexpr uint32_t A_SB = A_KQ + 16384 + 8192, A_SN = A_V + 8192, A_SE = A_V, A_SE2 = A_V, A_SG = A_SB;
static_assert(A_SB + 8192 == A_V && A_SE + 8192 == A_SN, "solve tiles and their row copies");
constexpr uint32_t A_ERR = 96;   // error flag, TMEM address and wait flag after the mbarriers
static_assert(A_NBARS * 8 <= A_ERR && A_ERR + 24 <= 128, "prep barrier block");

__global__ void __launch_bounds__(kAThreads, 3)
    chunk_prep_kernel(const SplitArgs a, int wave, int item0, int dep_wait, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = ptx::smem_align1024(smem_raw);
    Shared S;
    S.base = sm;
    S.bar = reinterpret_cast<uint64_t *>(sm + A_BAR);
    S.err = reinterpret_cast<volatile int *>(sm + A_BAR + A_ERR);
    S.tmem = reinterpret_cast<uint32_t *>(sm + A_BAR + A_ERR + 8);
    volatile int *wflag = reinterpret_cast<volatile int *>(sm + A_BAR + A_ERR + 16);
    float *gC = reinterpret_cast<float *>(sm + A_GC);
    float *bs = reinterpret_cast<float *>(sm + A_BS);
    float *pd = reinterpret_cast<float *>(sm + A_PD);
    float2 *red = reinterpret_cast<float2 *>(sm + A_RED);
    float *diag = reinterpret_cast<float *>(sm + A_DG);
    __nv_bfloat16 *halo = reinterpret_cast<__nv_bfloat16 *>(sm + A_HALO);

    // the chains of this wave may be placed (they wait for this grid to complete before
    // reading anything it writes) once every CTA of it has started
    ptx::grid_dep_launch();
    const PrefillArgs &pa = a.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = pa.H;
    const int e = blockIdx.x / H, h = blockIdx.x % H;
    const SplitItem it = a.items[item0 + e];
    const SeqMeta m = pa.seqs[it.seq];
    const int64_t start = m.start_pos, end = m.start_pos + m.len;
    const int64_t c_first = start / C;
    const int nchunks = (int)((end - 1) / C - c_first + 1);
    const int64_t abs0 = (c_first + it.lc) * C;
    const int r_first = start > abs0 ? (int)(start - abs0) : 0;
    const int r_end = end - abs0 < C ? (int)(end - abs0) : C;
    const uint64_t rec = (uint64_t)h * (uint64_t)pa.pool.rec_bytes;
    const int32_t *act_pages = pa.pages + m.active_off;
    uint8_t *img = image_addr(a, wave, e, h);
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(pa.q);
    const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(pa.k);
    const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(pa.v);
    const __nv_bfloat16 *betag = static_cast<const __nv_bfloat16 *>(pa.beta);

    if (tid == 128) {
        for (int i = 0; i < A_NBARS; ++i) ptx::mbar_init(&S.bar[i], 1);
        *S.err = 0;
        ptx::fence_mbar_init();
        // raw q, k, v, alpha tiles of the chunk (rows outside the sequence are masked later)
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_a);
        const int32_t y = it.row0;
        uint64_t *fb = &S.bar[AB_FULL];
        ptx::mbar_arrive_expect_tx(fb, 4 * 2 * 64 * 128);
        for (int kb = 0; kb < 2; ++kb) {
            const int32_t x = h * D + kb * 64;
            ptx::tma_load_2d(sm + A_KQ + kb * 16384, &tm_k, fb, x, y);
            ptx::tma_load_2d(sm + A_KQ + kb * 16384 + 8192, &tm_q, fb, x, y);
            ptx::tma_load_2d(sm + A_V + kb * 8192, &tm_v, fb, x, y);
            ptx::tma_load_2d(sm + A_AL + kb * 8192, &tm_a, fb, x, y);
        }
    }
    if (warp == 4) {
        ptx::tmem_alloc(S.tmem, 128);
        ptx::tmem_relinquish();
    }
    // Conv window before the first valid row (16 bytes per thread: raw tokens from the input,
    // or from the active object's window for positions before this call's start, or zeros)
    // and beta: loaded into registers now, stored to shared memory after the tile wait, so
    // that their latency overlaps the tile loads.
    const int64_t fv = abs0 + r_first;
    // 144 vectors of 8 channels (48 per token): compute thread t takes vector t and, for
    // t < 16, vector 128 + t
    auto load_halo = [&](int x) {
        uint4 val = make_uint4(0, 0, 0, 0);
        const int u = x / 48, c = (x - u * 48) * 8;
        const int64_t pos = fv - 3 + u;
        if (pos >= start) {
            const int64_t row = (int64_t)m.tok_begin + (pos - start);
            const __nv_bfloat16 *src = c < D ? qg : (c < 2 * D ? kg : vg);
            val = *reinterpret_cast<const uint4 *>(src + (row * H + h) * D + (c & (D - 1)));
        } else if (m.has_init) {
            const int slot = (int)(pos - start + 3);
            const uint4 *p = reinterpret_cast<const uint4 *>(obj_addr(
                pa.pool, act_pages, rec + (uint64_t)D * D * 4 + ((uint64_t)slot * 3 * D + c) * 2, pa.status));
            if (p) val = *p;
        }
        return val;
    };
    uint4 halo_v = make_uint4(0, 0, 0, 0), halo_w = make_uint4(0, 0, 0, 0);
    if (tid < 128) halo_v = load_halo(tid);
    if (tid < 16) halo_w = load_halo(128 + tid);
    __nv_bfloat16 beta_v = __float2bfloat16_rn(0.f);
    if (tid < C) {
        const int64_t pos = abs0 + tid;
        if (pos >= start && pos < end) beta_v = betag[((int64_t)m.tok_begin + (pos - start)) * H + h];
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = *S.tmem;

    if (warp == 4) {
        // ------------------------------------------------------------------ TMA / MMA / stores
        if (lane == 0) {
            bool m1 = false, m2 = false;
            const uint32_t sbase = ptx::smem_u32(sm);
            if (wait_bar(S, AB_P1, 0)) {
                // M1: G | P = [Kt'; Qt'] Kb^T
                ptx::tc_fence_after();
                const uint32_t id_gp = ptx::idesc_bf16(128, 64, 0, 0);
                for (int s = 0; s < 8; ++s) {
                    const uint64_t ad = ptx::sdesc_sw128(sbase + A_KQ + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                    const uint64_t bd = ptx::sdesc_sw128(sbase + A_AL + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024);
                    ptx::mma_bf16(tbase, ad, bd, id_gp, s > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&S.bar[AB_GP]);
                m1 = true;
                // Kb to the image: its tile becomes the solve scratch once M1 and this copy have
                // read it (KBF).  (V, q gamma_r and P^T go to the image from the compute
                // warps' registers.)
                ptx::bulk_store(img + IMG_PK + 8192, sm + A_AL, 16384);
                ptx::bulk_commit();
                ptx::bulk_wait_read0();
                if (wait_bar(S, AB_GP, 0)) ptx::mbar_arrive(&S.bar[AB_KBF]);
            }
            if (!*S.err && wait_bar(S, AB_T, 0)) {
                // M2: WK'^T = Kt'^T T^T (the chain forms U^T = V^T T^T itself, from V and T)
                ptx::tc_fence_after();
                const uint32_t id_m2 = ptx::idesc_bf16(128, 64, 1, 0);
                for (int s = 0; s < 4; ++s) {
                    const uint64_t bd = ptx::sdesc_sw128(sbase + A_T + s * 32, 16, 1024);
                    ptx::mma_bf16(tbase, ptx::sdesc_sw128(sbase + A_KQ + s * 2048, 16384, 1024), bd, id_m2,
                                  s > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&S.bar[AB_M2]);
                m2 = true;
                ptx::bulk_store(img + IMG_T, sm + A_T, 8192);
                ptx::bulk_commit();
            }
            // the image stores need only have read their shared memory before the CTA exits:
            // the grid's completion, which the chains wait for, covers their global writes
            ptx::bulk_wait_read0();
            if (*S.err) {
                // leave nothing in flight: the tile loads and any issued MMA
                uint32_t n = 0;
                while (!ptx::mbar_try_wait(&S.bar[AB_FULL], 0) && n < ptx::kSpinLimit) ++n;
                n = 0;
                while (m1 && !ptx::mbar_try_wait(&S.bar[AB_GP], 0) && n < ptx::kSpinLimit) ++n;
                n = 0;
                while (m2 && !ptx::mbar_try_wait(&S.bar[AB_M2], 0) && n < ptx::kSpinLimit) ++n;
            }
        }
    } else {
        // ------------------------------------------------------------------ compute warpgroup
        const int t = tid;                              // 0..127, TMEM lane
        const int p = t & 63, hf = t >> 6;              // channel pair (2p, 2p+1), row half
        const int c0 = 2 * p, kb = c0 >> 6, cb = (c0 & 63) * 2;
        const uint32_t lanes = (uint32_t)(warp * 32) << 16;
        int solve_stages = 0;   // stages of the tensor-core solve issued (by thread 0)
        do {
            // conv weights of the channel pair, tap by tap: (channel c0, channel c0 + 1)
            float2 wq[4], wk[4], wv[4];
            {
                const float4 *cw = reinterpret_cast<const float4 *>(pa.conv_w + (int64_t)h * 3 * D * 4);
                const float4 q0 = cw[c0], q1 = cw[c0 + 1], k0 = cw[D + c0], k1 = cw[D + c0 + 1];
                const float4 v0 = cw[2 * D + c0], v1 = cw[2 * D + c0 + 1];
                wq[0] = make_float2(q0.x, q1.x); wq[1] = make_float2(q0.y, q1.y);
                wq[2] = make_float2(q0.z, q1.z); wq[3] = make_float2(q0.w, q1.w);
                wk[0] = make_float2(k0.x, k1.x); wk[1] = make_float2(k0.y, k1.y);
                wk[2] = make_float2(k0.z, k1.z); wk[3] = make_float2(k0.w, k1.w);
                wv[0] = make_float2(v0.x, v1.x); wv[1] = make_float2(v0.y, v1.y);
                wv[2] = make_float2(v0.z, v1.z); wv[3] = make_float2(v0.w, v1.w);
            }
            *reinterpret_cast<uint4 *>(halo + t * 8) = halo_v;          // vector x at x * 8 elements
            if (t < 16) *reinterpret_cast<uint4 *>(halo + (128 + t) * 8) = halo_w;
            if (t < C) bs[t] = __bfloat162float(beta_v);
            if (!wg_wait(S, AB_FULL, 0, t, kAWg, wflag)) break;
            // ---------------- conv, decay, scaled operands (in place)
            uint8_t *const qrow = sm + A_KQ + kb * 16384 + 8192, *const krow = sm + A_KQ + kb * 16384;
            uint8_t *const vrow = sm + A_V + kb * 8192, *const arow = sm + A_AL + kb * 8192;
            float2 wqv[3], wkv[3], wvv[3];
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                wqv[u] = make_float2(__bfloat162float(halo[u * 384 + c0]), __bfloat162float(halo[u * 384 + c0 + 1]));
                wkv[u] = make_float2(__bfloat162float(halo[u * 384 + D + c0]), __bfloat162float(halo[u * 384 + D + c0 + 1]));
                wvv[u] = make_float2(__bfloat162float(halo[u * 384 + 2 * D + c0]),
                                     __bfloat162float(halo[u * 384 + 2 * D + c0 + 1]));
            }
            // the second half starts after the last (up to three) valid rows below row 32
            if (hf == 1) {
                const int hi = r_end < 32 ? r_end : 32;
                const int lo = (hi - 3) > r_first ? (hi - 3) : r_first;
                for (int r = lo; r < hi; ++r) {
                    const uint32_t off = ptx::sw128_off(r, cb);
                    const float2 xq = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qrow + off));
                    const float2 xk = bf2_to_f2(*reinterpret_cast<const uint32_t *>(krow + off));
                    const float2 xv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(vrow + off));
                    wqv[0] = wqv[1]; wqv[1] = wqv[2]; wqv[2] = xq;
                    wkv[0] = wkv[1]; wkv[1] = wkv[2]; wkv[2] = xk;
                    wvv[0] = wvv[1]; wvv[1] = wvv[2]; wvv[2] = xv;
                }
            }
            float2 ap[4] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f), make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) {
                const int r = hf * 32 + rr;
                const float2 al = bf2_to_f2(*reinterpret_cast<const uint32_t *>(arow + ptx::sw128_off(r, cb)));
                const bool valid = r >= r_first && r < r_end;
                ap[rr & 3].x *= valid ? al.x : 1.f;
                ap[rr & 3].y *= valid ? al.y : 1.f;
            }
            red[hf * 64 + p] = make_float2((ap[0].x * ap[1].x) * (ap[2].x * ap[3].x), (ap[0].y * ap[1].y) * (ap[2].y * ap[3].y));
            named_bar(kAWg, 128);
            const float2 h0 = red[p], h1 = red[64 + p];
            const float gCx = h0.x * h1.x, gCy = h0.y * h1.y;
            const float2 ic = make_float2(1.f / gCx, 1.f / gCy);
            if (hf == 0) {
                gC[c0] = gCx;
                gC[c0 + 1] = gCy;
                // the row scales gamma_r / gamma_C reach 1 / gamma_C: report a chunk whose
                // decay leaves the range they are exact in (NaN included)
                if (!(gCx >= kMinChunkDecay && gCy >= kMinChunkDecay)) flag_status(pa.status, KDA_DEV_RANGE);
            }
            float2 g2 = hf ? h0 : make_float2(1.f, 1.f);
            uint32_t swz[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) swz[u] = ptx::sw128_off(u, cb);
            // One row: conv, running decay, bf16 operands written in place (Kb over the alpha
            // tile); the pair-summed share of the diagonal q.k of the row goes to `diag`.
            auto row_proc = [&](int r, uint32_t off, float2 xq, float2 xk, float2 xv, float2 al, bool valid) {
                uint32_t oq = 0, ok = 0, okb = 0, ov = 0, oqg = 0;
                float dpart = 0.f;
                if (valid) {
                    float2 qb = fmul2(wq[0], wqv[0]), kbv = fmul2(wk[0], wkv[0]), vb = fmul2(wv[0], wvv[0]);
                    qb = ffma2(wq[1], wqv[1], qb);
                    kbv = ffma2(wk[1], wkv[1], kbv);
                    vb = ffma2(wv[1], wvv[1], vb);
                    qb = ffma2(wq[2], wqv[2], qb);
                    kbv = ffma2(wk[2], wkv[2], kbv);
                    vb = ffma2(wv[2], wvv[2], vb);
                    qb = ffma2(wq[3], xq, qb);
                    kbv = ffma2(wk[3], xk, kbv);
                    vb = ffma2(wv[3], xv, vb);
                    wqv[0] = wqv[1]; wqv[1] = wqv[2]; wqv[2] = xq;
                    wkv[0] = wkv[1]; wkv[1] = wkv[2]; wkv[2] = xk;
                    wvv[0] = wvv[1]; wvv[1] = wvv[2]; wvv[2] = xv;
                    g2 = fmul2(g2, al);
                    const float2 qk = fmul2(qb, kbv);
                    dpart = qk.x + qk.y;
                    const float2 s2 = fmul2(g2, ic);                  // gamma_r / gamma_C
                    const float2 qs = fmul2(qb, s2), ks = fmul2(kbv, s2);
                    const float2 kr = fmul2(kbv, make_float2(rcp_approx(s2.x), rcp_approx(s2.y)));
                    oq = pack_bf16x2(qs.x, qs.y);
                    const float2 qg = fmul2(qb, g2);                  // q gamma_r: the image's operand
                    oqg = pack_bf16x2(qg.x, qg.y);
                    ok = pack_bf16x2(ks.x, ks.y);
                    okb = pack_bf16x2(kr.x, kr.y);
                    ov = pack_bf16x2(vb.x, vb.y);
                }
                // sum over groups of four lanes (eight channels); 16 partials per row
                float dsum = dpart + __shfl_xor_sync(0xffffffffu, dpart, 1);
                dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
                if ((lane & 3) == 0) diag[r * 16 + (p >> 2)] = dsum;
                *reinterpret_cast<uint32_t *>(qrow + off) = oq;
                *reinterpret_cast<uint32_t *>(img + IMG_WQ + kb * 16384 + 8192 + off) = oqg;
                *reinterpret_cast<uint32_t *>(krow + off) = ok;
                *reinterpret_cast<uint32_t *>(arow + off) = okb;
                *reinterpret_cast<uint32_t *>(img + IMG_V + kb * 8192 + off) = ov;   // V: image only
            };
            if (r_first == 0 && r_end == C) {
#pragma unroll 1
                for (int r0 = hf * 32; r0 < hf * 32 + 32; r0 += 8) {
#pragma unroll
                    for (int h4 = 0; h4 < 8; h4 += 4) {
                        float2 xq[4], xk[4], xv[4], al[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t off = (uint32_t)(r0 + h4 + u) * 128u + (swz[h4 + u] & 127u);
                            xq[u] = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qrow + off));
                            xk[u] = bf2_to_f2(*reinterpret_cast<const uint32_t *>(krow + off));
                            xv[u] = bf2_to_f2(*reinterpret_cast<const uint32_t *>(vrow + off));
                            al[u] = bf2_to_f2(*reinterpret_cast<const uint32_t *>(arow + off));
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            row_proc(r0 + h4 + u, (uint32_t)(r0 + h4 + u) * 128u + (swz[h4 + u] & 127u), xq[u], xk[u],
                                     xv[u], al[u], true);
                    }
                }
            } else {
#pragma unroll 1
                for (int r = hf * 32; r < hf * 32 + 32; ++r) {
                    const uint32_t off = ptx::sw128_off((uint32_t)r, cb);
                    const float2 xq = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qrow + off));
                    const float2 xk = bf2_to_f2(*reinterpret_cast<const uint32_t *>(krow + off));
                    const float2 xv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(vrow + off));
                    const float2 al = bf2_to_f2(*reinterpret_cast<const uint32_t *>(arow + off));
                    row_proc(r, off, xq, xk, xv, al, r >= r_first && r < r_end);
                }
            }
            ptx::fence_proxy_async_smem();
            named_bar(kAWg, 128);
            if (t == 0) ptx::mbar_arrive(&S.bar[AB_P1]);
            // conv window after this chunk (the second half holds it)
            if (hf == 1) {
#pragma unroll
                for (int u = 0; u < 3; ++u) {
                    halo[u * 384 + c0] = __float2bfloat16_rn(wqv[u].x);
                    halo[u * 384 + c0 + 1] = __float2bfloat16_rn(wqv[u].y);
                    halo[u * 384 + D + c0] = __float2bfloat16_rn(wkv[u].x);
                    halo[u * 384 + D + c0 + 1] = __float2bfloat16_rn(wkv[u].y);
                    halo[u * 384 + 2 * D + c0] = __float2bfloat16_rn(wvv[u].x);
                    halo[u * 384 + 2 * D + c0 + 1] = __float2bfloat16_rn(wvv[u].y);
                }
            }
            // exact fp32 diagonal of P from the pair sums (rotated order: no bank conflicts)
            if (t < C) {
                float acc = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < 16; ++s2) acc += diag[t * 16 + ((s2 + t) & 15)];
                pd[t] = acc;
            }
            named_bar(kAWg, 128);
            {
                // window of a checkpoint ending here; the final window goes to the scratch
                const int ck = it.ckpt;
                const uint4 *src = reinterpret_cast<const uint4 *>(halo);
                if (ck >= 0) {
                    const int32_t *pg = pa.pages + pa.ckpts[ck].pages_off;
                    for (int x = t; x < 9 * D * 2 / 16; x += 128) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            obj_addr(pa.pool, pg, rec + (uint64_t)D * D * 4 + (uint64_t)x * 16, pa.status));
                        if (dst) *dst = src[x];
                    }
                }
                if (it.lc == nchunks - 1) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.win_scr + ((int64_t)it.seq * H + h) * (9 * D * 2));
                    for (int x = t; x < 9 * D * 2 / 16; x += 128) dst[x] = src[x];
                }
            }
            // ---------------- G | P from TMEM; A = Diag(beta) strict_lower(G) into the solve scratch
            if (!wg_wait(S, AB_GP, 0, t, kAWg, wflag)) break;
            if (!wg_wait(S, AB_KBF, 0, t, kAWg, wflag)) break;
            ptx::tc_fence_after();
            float *Msc = reinterpret_cast<float *>(sm + A_AL);
            {
                float g0[32], g1[32];
                ptx::tmem_ld32(tbase + lanes, g0);
                ptx::tmem_ld32(tbase + lanes + 32, g1);
                ptx::tmem_wait_ld();
                if (t < C) {
                    const int r = t;
                    const float br = bs[r];
                    float4 *row = reinterpret_cast<float4 *>(Msc + r * 64);
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        float ev[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int s2 = c4 * 4 + u;
                            const float gv = s2 < 32 ? g0[s2 & 31] : g1[s2 & 31];
                            ev[u] = s2 < r ? br * gv : 0.f;
                        }
                        row[c4 ^ (r & 7)] = make_float4(ev[0], ev[1], ev[2], ev[3]);
                    }
                } else {
                    // P^T straight from the registers into the image, MN-major and swizzled as
                    // the chain reads it: row j holds P[0..63][j]; thread r writes column r
                    // (a warp's store fills whole 32-byte sectors of one row)
                    const int r = t - C;
                    const float pdr = pd[r];
                    uint8_t *const pt = img + IMG_PK;
#pragma unroll
                    for (int s0 = 0; s0 < 64; ++s0) {
                        const float gv = s0 < 32 ? g0[s0 & 31] : g1[s0 & 31];
                        *reinterpret_cast<__nv_bfloat16 *>(pt + ptx::sw128_off(s0, (uint32_t)r * 2)) =
                            __float2bfloat16_rn(s0 < r ? gv : (s0 == r ? pdr : 0.f));
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            named_bar(kAWg, 128);
            // Each stage: the compute warps write its operands, meet at a barrier, and thread 0
            // issues the stage's MMAs and its commit; the stage's completion is polled by
            // thread 0 and handed to the warpgroup through a flag word of its own (one barrier).
            volatile int *solve_flag = reinterpret_cast<volatile int *>(sm + A_RED);   // free after the conv
            auto solve_issue = [&](int rd) {
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                named_bar(kAWg, 128);
                if (t == 0) {
                    ptx::tc_fence_after();
                    const uint32_t sbase = ptx::smem_u32(sm);
                    const uint32_t id64 = ptx::idesc_bf16(128, 64, 0, 1);
                    // one N = 64 product into TMEM columns d_col..+63; K-steps (16-row blocks of
                    // the shared dimension) whose products are all zero are skipped: N and E have
                    // no entries in their first row block, E none in its last column block, E^2
                    // none in its last two
                    auto product = [&](uint32_t d_col, uint32_t a_t, uint32_t b_t, int s0, int s1) {
                        for (int s = s0; s < s1; ++s)
                            ptx::mma_bf16(tbase + d_col, ptx::sdesc_sw128(sbase + a_t + s * 32, 16, 1024),
                                          ptx::sdesc_sw128(sbase + b_t + s * 2048, 8192, 1024), id64, s > s0 ? 1u : 0u);
                    };
                    if (rd == 0) {
                        product(0, A_SB, A_SN, 1, 4);        // E = Binv N
                    } else if (rd == 1) {
                        product(0, A_SE, A_SE, 1, 3);        // E^2
                        product(64, A_SE, A_SB, 0, 3);       // E Binv
                    } else {
                        product(0, A_SE2, A_SG, 0, 2);       // E^2 G
                    }
                    ptx::mma_commit(&S.bar[AB_SO]);
                }
                solve_stages = rd + 1;
            };
            auto solve_wait = [&](int rd) -> bool {
                if (t == 0) solve_flag[rd] = ptx::mbar_wait(&S.bar[AB_SO], (uint32_t)(rd & 1), S.err) ? 1 : 0;
                named_bar(kAWg, 128);
                return solve_flag[rd] != 0;
            };
            auto put_row_bf16 = [&](uint32_t tile, int r, int ch0, const float *v8x4) {   // 4 units of 8
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 pk;
                    pk.x = pack_bf16x2(v8x4[j * 8 + 0], v8x4[j * 8 + 1]);
                    pk.y = pack_bf16x2(v8x4[j * 8 + 2], v8x4[j * 8 + 3]);
                    pk.z = pack_bf16x2(v8x4[j * 8 + 4], v8x4[j * 8 + 5]);
                    pk.w = pack_bf16x2(v8x4[j * 8 + 6], v8x4[j * 8 + 7]);
                    *reinterpret_cast<uint4 *>(sm + tile + ptx::sw128_off(r, (ch0 + j) * 16)) = pk;
                }
            };
            // ---------------- T = (I + A)^{-1} Diag(beta)
            // level 0: the four 16 x 16 diagonal blocks, one row per thread (from the last row up)
            if (t < C) {
                const int r = t, bb = r >> 4, rr = r & 15;
                float x[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) x[c] = c == rr ? 1.f : 0.f;
#pragma unroll
                for (int mm = 15; mm >= 1; --mm) {
                    const int ar = bb * 16 + mm;
                    const float4 *arow4 = reinterpret_cast<const float4 *>(Msc + ar * 64);
                    float av[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (q * 4 < mm) {
                            const float4 v4 = arow4[(bb * 4 + q) ^ (ar & 7)];
                            av[q * 4] = v4.x; av[q * 4 + 1] = v4.y; av[q * 4 + 2] = v4.z; av[q * 4 + 3] = v4.w;
                        }
                    }
                    const float xm = x[mm];
#pragma unroll
                    for (int c = 0; c < mm; ++c) x[c] = fmaf(-xm, av[c], x[c]);
                }
                named_bar(kAHalf, 64);
                float4 *row = reinterpret_cast<float4 *>(Msc + r * 64);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    row[(bb * 4 + q) ^ (r & 7)] = make_float4(x[q * 4], x[q * 4 + 1], x[q * 4 + 2], x[q * 4 + 3]);
                // the row of Binv as bf16 (its 16-column block, zeros elsewhere)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 pk = make_uint4(0, 0, 0, 0);
                    if ((ch >> 1) == bb) {
                        const float *xs = x + (ch & 1) * 8;
                        pk.x = pack_bf16x2(xs[0], xs[1]);
                        pk.y = pack_bf16x2(xs[2], xs[3]);
                        pk.z = pack_bf16x2(xs[4], xs[5]);
                        pk.w = pack_bf16x2(xs[6], xs[7]);
                    }
                    *reinterpret_cast<uint4 *>(sm + A_SB + ptx::sw128_off(r, ch * 16)) = pk;
                    *reinterpret_cast<uint4 *>(sm + A_SB + 8192 + ptx::sw128_off(r, ch * 16)) = pk;   // rows 64-127
                }
            } else {
                // meanwhile: N, the strictly block-lower part of A (untouched by level 0), as bf16,
                // over the second half of the raw v tile
                const int r = t - C, rb = r >> 4;
                const float4 *row = reinterpret_cast<const float4 *>(Msc + r * 64);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 pk = make_uint4(0, 0, 0, 0);
                    if ((ch >> 1) < rb) {
                        const float4 m0 = row[(ch * 2) ^ (r & 7)], m1 = row[(ch * 2 + 1) ^ (r & 7)];
                        pk.x = pack_bf16x2(m0.x, m0.y);
                        pk.y = pack_bf16x2(m0.z, m0.w);
                        pk.z = pack_bf16x2(m1.x, m1.y);
                        pk.w = pack_bf16x2(m1.z, m1.w);
                    }
                    *reinterpret_cast<uint4 *>(sm + A_SN + ptx::sw128_off(r, ch * 16)) = pk;
                }
            }
            // Off-diagonal part on the tensor cores: with Binv = the block-diagonal inverse and N
            // the strictly block-lower part of A, L = I + A has L^{-1} = (I - E)(I + E^2) Binv =
            // G + E^2 G, E = Binv N, G = Binv - E Binv (E^4 = 0).  Three bf16 MMA stages with
            // fp32 accumulation: E = Binv N; E^2 and E Binv; E^2 G (10 MMAs: the block structure
            // leaves some 16-deep steps of each product zero).  Every operand is a 64 x 64 bf16
            // tile, row-major and 128-byte swizzled, which serves as a K-major A and as an
            // MN-major B alike.  Thread t takes row t % 64 and column half t / 64 of each
            // product, from the TMEM lanes of its warp (lanes 64-127 repeat rows 0-63).
            const int sr = t & 63, shf = t >> 6;
            solve_issue(0);
            // stage 1 done: E -> bf16 tile and its row copy
            if (!solve_wait(0)) break;
            ptx::tc_fence_after();
            {
                float e[32];
                ptx::tmem_ld32(tbase + lanes + shf * 32, e);
                ptx::tmem_wait_ld();
                put_row_bf16(A_SE, sr, shf * 4, e);
                put_row_bf16(A_SE + 8192, sr, shf * 4, e);
            }
            solve_issue(1);
            // stage 2 done: E^2 -> bf16 tile and copy; G = Binv - E Binv -> bf16 tile and fp32 row of Msc
            if (!solve_wait(1)) break;
            ptx::tc_fence_after();
            {
                const int r = sr, rb = r >> 4;
                float4 *row = reinterpret_cast<float4 *>(Msc + r * 64);
                float e2[32], eb[32];
                ptx::tmem_ld32(tbase + lanes + shf * 32, e2);
                ptx::tmem_ld32(tbase + lanes + 64 + shf * 32, eb);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const int cc = shf * 8 + c4;
                    float4 g4 = make_float4(-eb[c4 * 4], -eb[c4 * 4 + 1], -eb[c4 * 4 + 2], -eb[c4 * 4 + 3]);
                    if ((cc >> 2) == rb) {
                        const float4 b4 = row[cc ^ (r & 7)];
                        g4.x += b4.x; g4.y += b4.y; g4.z += b4.z; g4.w += b4.w;
                    }
                    eb[c4 * 4] = g4.x; eb[c4 * 4 + 1] = g4.y; eb[c4 * 4 + 2] = g4.z; eb[c4 * 4 + 3] = g4.w;
                }
                // Binv of this half read above; G overwrites it (only this thread uses it)
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                    row[(shf * 8 + c4) ^ (r & 7)] = make_float4(eb[c4 * 4], eb[c4 * 4 + 1], eb[c4 * 4 + 2], eb[c4 * 4 + 3]);
                put_row_bf16(A_SE2, r, shf * 4, e2);
                put_row_bf16(A_SE2 + 8192, r, shf * 4, e2);
                put_row_bf16(A_SG, r, shf * 4, eb);
            }
            solve_issue(2);
            // stage 3 done: T = (G + E^2 G) Diag(beta), lower triangle, as the bf16 operand
            if (!solve_wait(2)) break;
            ptx::tc_fence_after();
            {
                const int r = sr;
                const float4 *row = reinterpret_cast<const float4 *>(Msc + r * 64);
                const float4 *b4 = reinterpret_cast<const float4 *>(bs);
                float d[32];
                ptx::tmem_ld32(tbase + lanes + shf * 32, d);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const int cc = shf * 8 + c4;
                    const float4 g4 = row[cc ^ (r & 7)], bv = b4[cc];
                    d[c4 * 4 + 0] = cc * 4 + 0 <= r ? (g4.x + d[c4 * 4 + 0]) * bv.x : 0.f;
                    d[c4 * 4 + 1] = cc * 4 + 1 <= r ? (g4.y + d[c4 * 4 + 1]) * bv.y : 0.f;
                    d[c4 * 4 + 2] = cc * 4 + 2 <= r ? (g4.z + d[c4 * 4 + 2]) * bv.z : 0.f;
                    d[c4 * 4 + 3] = cc * 4 + 3 <= r ? (g4.w + d[c4 * 4 + 3]) * bv.w : 0.f;
                }
                put_row_bf16(A_T, r, shf * 4, d);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            named_bar(kAWg, 128);
            if (t == 0) ptx::mbar_arrive(&S.bar[AB_T]);
            // ---------------- -WK' Gamma_C (K-major bf16 operand rows) and gamma_C, straight into the image
            if (!wg_wait(S, AB_M2, 0, t, kAWg, wflag)) break;
            ptx::tc_fence_after();
            {
                float w0[32], w1[32];
                ptx::tmem_ld32(tbase + lanes, w0);
                ptx::tmem_ld32(tbase + lanes + 32, w1);
                ptx::tmem_wait_ld();
                // thread t holds column t (key t) of WK'; row c of the K-major tile of key block
                // t / 64 gets it at position t % 64, negated (the chain accumulates -(Gamma S)^T WK'^T)
                uint8_t *const wk = img + IMG_WQ + (t >> 6) * 16384;
                const uint32_t cb2 = (uint32_t)(t & 63) * 2;
                const float gt = gC[t];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    *reinterpret_cast<__nv_bfloat16 *>(wk + ptx::sw128_off(c, cb2)) = __float2bfloat16_rn(-w0[c] * gt);
                    *reinterpret_cast<__nv_bfloat16 *>(wk + ptx::sw128_off(32 + c, cb2)) = __float2bfloat16_rn(-w1[c] * gt);
                }
                reinterpret_cast<float *>(img + IMG_GC)[t] = gC[t];
            }
        } while (false);
        // on a timeout, leave no solve MMA in flight: its commit tracks every MMA before it
        if (t == 0 && *S.err && solve_stages > 0) {
            uint32_t k = 0;
            while (!ptx::mbar_try_wait(&S.bar[AB_SO], (uint32_t)((solve_stages - 1) & 1)) && k < ptx::kSpinLimit) ++k;
        }
    }
    // ---------------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (*S.err && tid == 0) flag_status(pa.status, KDA_DEV_TIMEOUT);
    if (warp == 4) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, 128);
    }
    // launched beside the chains of the previous wave: this grid completes only after them
    if (dep_wait && blockIdx.x == gridDim.x - 1) ptx::grid_dep_wait();
}

// ============================================================================ chain
// 16 warps: warp 0 loads images, warp 1 issues MMAs, warp 2 stages the wave's checkpoint
// page lists, warps 4-7 and 8-11 run the state epilogues on the low and high halves of the
// key columns, warps 12-15 write the outputs; warp 3 idles.
constexpr int kBThreads = 512;
constexpr uint32_t B_SLOT = (kImageBytes + 1023) / 1024 * 1024;   // image slot stride
constexpr uint32_t B_WT = 2 * B_SLOT;            // [128 rows][128 B] W^T bf16 (A operand)
constexpr uint32_t B_OST = B_WT + 16384;         // [64 rows][256 B] bf16 output staging
constexpr uint32_t B_PGL = B_OST + 16384;        // int32 [kPglCap]: page lists of this wave's checkpoints
constexpr int kPglCap = 1024;
constexpr uint32_t B_BAR = B_PGL + kPglCap * 4;
constexpr int kBPgl = 2;   // named barrier: page-list copy (warp 2) -> state warps
constexpr uint32_t B_SMEM = B_BAR + 256 + 1024;
constexpr int kBOut = 1;   // named barrier of the output warpgroup

// TMEM columns: W^T | O^T | S^T (64 + 64 + 128), adjacent so that one N = 128 MMA group forms
// W^T = U^T - (Gamma S)^T WK'^T with the first half of O^T, and one N = 192 group the second
// half of O^T with the state update; then bf16 (Gamma S)^T (two buffers, two values per column).
constexpr uint32_t COL_W = 0, COL_O = 64, COL_S = 128, COL_SA = 256;

// mbarriers ([2] by chunk parity).  SB and WT count the 8 state warps, DO the 4 output warps.
enum {
    BB_FULL = 0,    // image landed (tx)
    BB_SB = 2,      // (Gamma S)^T written, S scaled
    BB_W = 4,       // W^T (and the first half of O^T) in TMEM
    BB_WT = 6,      // W^T operand written
    BB_M4S = 8,     // every MMA of the chunk done: S advanced, O^T complete, image slot free
    BB_DO = 10,     // O^T read and zeroed (one buffer: counts chunks)
    BB_DRAIN = 11,  // error path: every issued MMA done
    B_NBARS = 12
};

// First checkpoint of sequence m at or after position pos (index relative to the sequence).
__device__ __forceinline__ int lower_ckpt(const PrefillArgs &a, const SeqMeta &m, int64_t pos) {
    int lo = 0, hi = m.ckpt_count;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a.ckpts[m.ckpt_begin + mid].pos < pos) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kBThreads, 1) chain_kernel(const SplitArgs a, int wave, int lc0w, int lc1w) {
    const PrefillArgs &pa = a.p;
    const int H = pa.H;
    const int h = blockIdx.x % H, sq = blockIdx.x / H;
    const SeqMeta m = pa.seqs[sq];
    const int64_t start = m.start_pos, end = m.start_pos + m.len;
    const int64_t c_first = start / C;
    const int nchunks = m.len > 0 ? (int)((end - 1) / C - c_first + 1) : 0;
    const uint64_t rec = (uint64_t)h * (uint64_t)pa.pool.rec_bytes;
    const int32_t *act_pages = pa.pages + m.active_off;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (nchunks == 0) {
        // empty sequence: a fresh one gets a zero state and window, a resumed one keeps its own
        ptx::grid_dep_wait();
        if (wave == 0 && !m.has_init) {
            for (int x = tid; x < (D * D * 4 + 9 * D * 2) / 16; x += kBThreads) {
                uint4 *dst = reinterpret_cast<uint4 *>(obj_addr(pa.pool, act_pages, rec + (uint64_t)x * 16, pa.status));
                if (dst) *dst = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int lc0 = lc0w;
    if (lc0 >= nchunks) return;
    const int lc1 = lc1w < nchunks ? lc1w : nchunks;
    const int cnt = lc1 - lc0;
    const bool first = lc0 == 0, last = lc1 == nchunks;
    const int32_t off0 = a.wave_seq_off[(int64_t)wave * pa.nseq + sq];
    if (off0 < 0) {
        if (tid == 0) flag_status(pa.status, KDA_DEV_BAD_META);
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = ptx::smem_align1024(smem_raw);
    Shared S;
    S.base = sm;
    S.bar = reinterpret_cast<uint64_t *>(sm + B_BAR);
    S.err = reinterpret_cast<volatile int *>(sm + B_BAR + B_NBARS * 8);
    S.tmem = reinterpret_cast<uint32_t *>(sm + B_BAR + B_NBARS * 8 + 16);
    // Checkpoints of this wave (positions in ((c_first + lc0) C, (c_first + lc1) C]): their page
    // lists are copied to shared memory by warp 2 while the state warps load the state, so a
    // checkpoint store never waits on a global page-list load; more than fit: read in place.
    const int ck_lo = lower_ckpt(pa, m, (c_first + lc0) * C + 1), ck_hi = lower_ckpt(pa, m, (c_first + lc1) * C + 1);
    const int P = pa.pool.pages_per_object;
    const bool pgl_smem = (ck_hi - ck_lo) * P <= kPglCap;
    int32_t *pgl = reinterpret_cast<int32_t *>(sm + B_PGL);
    auto ck_pages = [&](int ck) -> const int32_t * {   // ck: index within the sequence
        return pgl_smem ? pgl + (ck - ck_lo) * P : pa.pages + pa.ckpts[m.ckpt_begin + ck].pages_off;
    };

    if (tid == 0) {
        for (int i = 0; i < B_NBARS; ++i) {
            const uint32_t cntw = (i == BB_SB || i == BB_SB + 1 || i == BB_WT || i == BB_WT + 1) ? 8u
                                  : i == BB_DO ? 4u : 1u;
            ptx::mbar_init(&S.bar[i], cntw);
        }
        *S.err = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(S.tmem, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = *S.tmem;
    // launched while the chunk prep of this wave (and through it the chains of the previous
    // wave) may still run: nothing they write is read before this point.  Only then may the
    // next wave's prep be placed: it overwrites the image slot that the chains two waves
    // back read, and those are complete once this wave's prep is.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();

    if (warp == 0) {
        // ------------------------------------------------------------------ image loads
        if (lane == 0) {
            int issued = 0;
            for (int n = 0; n < cnt && !*S.err; ++n) {
                const int b = n & 1;
                if (n >= 2 && !wait_bar(S, BB_M4S + b, par(n - 2))) break;   // slot consumed
                ptx::mbar_arrive_expect_tx(&S.bar[BB_FULL + b], (uint32_t)kImageBytes);
                ptx::bulk_load(sm + b * B_SLOT, image_addr(a, wave, off0 + n, h), (uint32_t)kImageBytes,
                               &S.bar[BB_FULL + b]);
                ++issued;
            }
            if (*S.err)
                for (int n = 0; n < issued; ++n) {
                    uint32_t k = 0;
                    while (!ptx::mbar_try_wait(&S.bar[BB_FULL + (n & 1)], par(n)) && k < ptx::kSpinLimit) ++k;
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_wq = ptx::idesc_bf16(128, 128, 0, 0);
            const uint32_t id_sp = ptx::idesc_bf16(128, 192, 0, 1);
            const uint32_t id_u = ptx::idesc_bf16(128, 64, 1, 0);
            const uint32_t sbase = ptx::smem_u32(sm), wt = sbase + B_WT;
            // Per chunk, in this order, each group after a blocking (bounded) wait on what it
            // needs: [W^T | O^T] += S^T (Gamma_C [-WK' | Qt'])^T (needs the bf16 state and the
            // emptied O^T; W^T accumulates onto U^T, O^T onto zeros), then [O^T | S^T] +=
            // W^T [P^T | Kb] (needs W^T), then U^T = V^T T^T of the next chunk into the W columns
            // (which E2 has read).  Every MMA holds the tensor pipe about the same time whatever
            // its N up to 128, so the groups are as wide and as few as the data allow.
            auto issue_u = [&](int n) {
                const uint32_t im = sbase + (n & 1) * B_SLOT;
                ptx::tc_fence_after();
                for (int s = 0; s < 4; ++s)
                    ptx::mma_bf16(tbase + COL_W, ptx::sdesc_sw128(im + IMG_V + s * 2048, 8192, 1024),
                                  ptx::sdesc_sw128(im + IMG_T + s * 32, 16, 1024), id_u, s > 0 ? 1u : 0u);
            };
            for (int n = 0; n < cnt; ++n) {
                const int b = n & 1;
                const uint32_t im = sbase + b * B_SLOT;
                if (n == 0) {
                    if (!wait_bar(S, BB_FULL, 0)) break;
                    issue_u(0);
                }
                if (!wait_bar(S, BB_DO, (uint32_t)(n & 1)) || !wait_bar(S, BB_SB + b, par(n))) break;
                // [W^T | O^T] += S^T (Gamma_C [-WK' | Qt'])^T
                ptx::tc_fence_after();
                for (int s = 0; s < 8; ++s) {
                    const uint64_t bq = ptx::sdesc_sw128(im + IMG_WQ + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                    ptx::mma_bf16_ta(tbase + COL_W, tbase + COL_SA + b * 64 + s * 8, bq, id_wq, 1u);
                }
                ptx::mma_commit(&S.bar[BB_W + b]);
                if (!wait_bar(S, BB_WT + b, par(n))) break;
                // [O^T | S^T] += W^T [P^T | Kb]
                ptx::tc_fence_after();
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ad = ptx::sdesc_sw128(wt + s * 32, 16, 1024);
                    const uint64_t bd = ptx::sdesc_sw128(im + IMG_PK + s * 2048, 8192, 1024);
                    ptx::mma_bf16(tbase + COL_O, ad, bd, id_sp, 1u);
                }
                ptx::mma_commit(&S.bar[BB_M4S + b]);   // frees this image slot for chunk n + 2
                if (n + 1 < cnt) {
                    if (!wait_bar(S, BB_FULL + (b ^ 1), par(n + 1))) break;
                    issue_u(n + 1);
                }
            }
            // leave no MMA in flight: one more commit tracks every MMA issued so far
            if (*S.err) {
                ptx::mma_commit(&S.bar[BB_DRAIN]);
                uint32_t k = 0;
                while (!ptx::mbar_try_wait(&S.bar[BB_DRAIN], 0) && k < ptx::kSpinLimit) ++k;
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------ checkpoint page lists
        if (pgl_smem && ck_hi > ck_lo) {
            for (int x = lane; x < (ck_hi - ck_lo) * P; x += 32) {
                const int k = x / P;
                pgl[x] = pa.pages[pa.ckpts[m.ckpt_begin + ck_lo + k].pages_off + (x - k * P)];
            }
            named_bar(kBPgl, 32 * 9);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------------ state epilogues
        const int g = (warp - 4) >> 2;                 // column half
        const int j = (warp & 3) * 32 + lane;          // value channel = TMEM lane
        const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
        const int ib = g * 64;                         // key channels [ib, ib + 64) of S^T
        float *scr = a.state_scr + ((int64_t)sq * H + h) * D * D;
        // state at the start of this wave, 32 loads in flight per batch
#pragma unroll 1
        for (int i0 = ib; i0 < ib + 64; i0 += 32) {
            float v[32];
            const uint64_t o0 = rec + ((uint64_t)i0 * D + j) * 4;
            const uint8_t *run = first && m.has_init ? run_addr(pa.pool, act_pages, o0, 31 * D * 4, pa.status) : nullptr;
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                float x = 0.f;
                if (!first) {
                    x = scr[(i0 + ii) * D + j];
                } else if (run) {
                    x = *reinterpret_cast<const float *>(run + ii * D * 4);
                } else if (m.has_init) {
                    const float *p = reinterpret_cast<const float *>(
                        obj_addr(pa.pool, act_pages, o0 + (uint64_t)ii * D * 4, pa.status));
                    if (p) x = *p;
                }
                v[ii] = x;
            }
            ptx::tmem_st32(tbase + lanes + COL_S + i0, v);
        }
        ptx::tmem_wait_st();
        if (pgl_smem && ck_hi > ck_lo) named_bar(kBPgl, 32 * 9);   // page lists copied
        // next checkpoint at or after the first chunk boundary of this wave
        int ck_i = ck_lo, pf_i = -1;   // next checkpoint; the last one prefetched
        int64_t ck_pos = ck_i < m.ckpt_count ? pa.ckpts[m.ckpt_begin + ck_i].pos : INT64_MAX;
        // this half of S (fp32, from TMEM) into the checkpoint at `pos` if there is one, into
        // the active object (final) or into the wave scratch (to_scratch)
        // 8 rows of column j (offsets o0 + 512 ii) of an object
        auto store_rows = [&](const int32_t *pgs, uint64_t o0, const float (&v)[8]) {
            uint8_t *run = run_addr(pa.pool, pgs, o0, 7 * D * 4, pa.status);
            if (run) {
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) *reinterpret_cast<float *>(run + ii * D * 4) = v[ii];
            } else {
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) {
                    float *dst = reinterpret_cast<float *>(obj_addr(pa.pool, pgs, o0 + (uint64_t)ii * D * 4, pa.status));
                    if (dst) *dst = v[ii];
                }
            }
        };
        auto write_state = [&](int64_t pos, bool final_state, bool to_scratch) {
            const bool hit = ck_pos == pos;
            if (!hit && !final_state && !to_scratch) return;
            const int32_t *pg = hit ? ck_pages(ck_i) : nullptr;
#pragma unroll 1
            for (int i0 = ib; i0 < ib + 64; i0 += 8) {
                float v[8];
                ptx::tmem_ld8(tbase + lanes + COL_S + i0, v);
                ptx::tmem_wait_ld();
                const uint64_t o0 = rec + ((uint64_t)i0 * D + j) * 4;
                if (pg) store_rows(pg, o0, v);
                if (final_state) store_rows(act_pages, o0, v);
                if (to_scratch) {
#pragma unroll
                    for (int ii = 0; ii < 8; ++ii) scr[(i0 + ii) * D + j] = v[ii];
                }
            }
            if (hit) {
                ++ck_i;
                ck_pos = ck_i < m.ckpt_count ? pa.ckpts[m.ckpt_begin + ck_i].pos : INT64_MAX;
            }
        };
        bool ok = true;
        for (int n = 0; n < cnt; ++n) {
            const int b = n & 1;
            // ---------------- E1: checkpoint S, bf16 operand S^T, then Gamma_C S in TMEM
            // A checkpoint at this chunk boundary is stored from the registers E1 loads S into: no
            // separate pass over S on the chain's critical path.  The decay Gamma_C is folded
            // into the image's first operand, so this part needs nothing from the image.
            const int32_t *ckpg = nullptr;
            if (n >= 1) {
                if (!(ok = warp_wait(S, BB_M4S + ((n - 1) & 1), par(n - 1)))) break;
                ptx::tc_fence_after();
                if (ck_pos == (c_first + lc0 + n) * C) {
                    ckpg = ck_pages(ck_i);
                    ++ck_i;
                    ck_pos = ck_i < m.ckpt_count ? pa.ckpts[m.ckpt_begin + ck_i].pos : INT64_MAX;
                }
            }
#pragma unroll 1
            for (int i0 = 0; i0 < 64; i0 += 32) {
                float v[32], pk[16];
                ptx::tmem_ld32(tbase + lanes + COL_S + ib + i0, v);
                ptx::tmem_wait_ld();
                if (ckpg) {
                    const uint64_t o0 = rec + ((uint64_t)(ib + i0) * D + j) * 4;
                    uint8_t *run = run_addr(pa.pool, ckpg, o0, 31 * D * 4, pa.status);
                    if (run) {
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) *reinterpret_cast<float *>(run + ii * D * 4) = v[ii];
                    } else {
#pragma unroll
                        for (int ii = 0; ii < 32; ++ii) {
                            float *dst = reinterpret_cast<float *>(obj_addr(pa.pool, ckpg, o0 + (uint64_t)ii * D * 4, pa.status));
                            if (dst) *dst = v[ii];
                        }
                    }
                }
#pragma unroll
                for (int q2 = 0; q2 < 16; ++q2) pk[q2] = __uint_as_float(pack_bf16x2(v[2 * q2], v[2 * q2 + 1]));
                ptx::tmem_st16(tbase + lanes + COL_SA + b * 64 + ((ib + i0) >> 1), pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            warp_arrive(&S.bar[BB_SB + b]);
            if (!(ok = warp_wait(S, BB_FULL + b, par(n)))) break;
            const float *gcb = reinterpret_cast<const float *>(sm + b * B_SLOT + IMG_GC);
            // S <- Gamma_C S in fp32 while the MMAs form W: the state update reads it only after
            // E2 below, which these stores precede
#pragma unroll 1
            for (int i0 = 0; i0 < 64; i0 += 32) {
                float v[32];
                ptx::tmem_ld32(tbase + lanes + COL_S + ib + i0, v);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) v[ii] *= gcb[ib + i0 + ii];
                ptx::tmem_st32(tbase + lanes + COL_S + ib + i0, v);
            }
            ptx::tmem_wait_st();
            // ---------------- E2: W^T (U^T with D_W accumulated) -> bf16 operand (chunk rows [32 g, 32 g + 32))
            if (!(ok = warp_wait(S, BB_W + b, par(n)))) break;
            ptx::tc_fence_after();
            {
                const int r0 = g * 32;
                float v[32];
                ptx::tmem_ld32(tbase + lanes + COL_W + r0, v);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint4 pk;
                    uint32_t *pp = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        pp[q2] = pack_bf16x2(v[ch * 8 + 2 * q2], v[ch * 8 + 2 * q2 + 1]);
                    }
                    *reinterpret_cast<uint4 *>(sm + B_WT + ptx::sw128_off(j, r0 * 2 + ch * 16)) = pk;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            warp_arrive(&S.bar[BB_WT + b]);
            // The next checkpoint's record into L2 a few chunks before E1 stores it there (its
            // first touch otherwise stalls those stores): two lines per state thread.
            if (ck_i < ck_hi && ck_i != pf_i && ck_pos <= (c_first + lc0 + n + 4) * C) {
                pf_i = ck_i;
                const int32_t *pg = ck_pages(ck_i);
                const int st = (warp - 4) * 32 + lane;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint8_t *q = obj_addr(pa.pool, pg, rec + (uint64_t)(st + 256 * u) * 128, pa.status);
                    if (q) ptx::prefetch_l2(q);
                }
            }
        }
        if (ok && warp_wait(S, BB_M4S + ((cnt - 1) & 1), par(cnt - 1))) {
            ptx::tc_fence_after();
            if (last) {
                write_state(end, true, false);
                // final conv window (written by the chunk-prep kernel) into the active object
                const uint4 *src = reinterpret_cast<const uint4 *>(a.win_scr + ((int64_t)sq * H + h) * (9 * D * 2));
                for (int x = tid - 128; x < 9 * D * 2 / 16; x += 256) {
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        obj_addr(pa.pool, act_pages, rec + (uint64_t)D * D * 4 + (uint64_t)x * 16, pa.status));
                    if (dst) *dst = src[x];
                }
            } else {
                write_state((c_first + lc1) * C, false, true);
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------------ outputs
        const int j = (warp & 3) * 32 + lane;
        const int jt = tid - 384;
        const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
        __nv_bfloat16 *ost = reinterpret_cast<__nv_bfloat16 *>(sm + B_OST);
        const __nv_bfloat16 *og0 = static_cast<const __nv_bfloat16 *>(pa.o);
        // The first MMA group of a chunk accumulates O^T onto its buffer: both buffers start
        // zeroed, and each is zeroed again once read.
        float zero[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
        ptx::tmem_st32(tbase + lanes + COL_O, zero);
        ptx::tmem_st32(tbase + lanes + COL_O + 32, zero);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        warp_arrive(&S.bar[BB_DO]);
        for (int n = 0; n < cnt; ++n) {
            const int b = n & 1;
            if (!warp_wait(S, BB_M4S + b, par(n))) break;
            ptx::tc_fence_after();
            float v0[32], v1[32];
            ptx::tmem_ld32(tbase + lanes + COL_O, v0);
            ptx::tmem_ld32(tbase + lanes + COL_O + 32, v1);
            ptx::tmem_wait_ld();
            ptx::tmem_st32(tbase + lanes + COL_O, zero);
            ptx::tmem_st32(tbase + lanes + COL_O + 32, zero);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            warp_arrive(&S.bar[BB_DO]);
            // transpose through shared memory: row r of the chunk = 128 channels (256 B)
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                ost[r * D + j] = __float2bfloat16_rn(v0[r]);
                ost[(32 + r) * D + j] = __float2bfloat16_rn(v1[r]);
            }
            named_bar(kBOut, 128);
            const int64_t abs0 = (c_first + lc0 + n) * C;
            const int r_first = start > abs0 ? (int)(start - abs0) : 0;
            const int r_end = end - abs0 < C ? (int)(end - abs0) : C;
            const int64_t row0 = (int64_t)m.tok_begin + (abs0 - start);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int x = jt + 128 * k, r = x >> 4, vc = x & 15;
                if (r >= r_first && r < r_end) {
                    uint4 *dst = reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(og0) +
                                                           ((row0 + r) * H + h) * D + vc * 8);
                    *dst = *reinterpret_cast<const uint4 *>(ost + r * D + vc * 8);
                }
            }
            named_bar(kBOut, 128);
        }
    }
    // ---------------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (*S.err && tid == 0) flag_status(pa.status, KDA_DEV_TIMEOUT);
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, 512);
    }
}

}  // namespace

cudaError_t launch_prefill_split(const SplitArgs &a, const SplitPlan &plan, cudaStream_t s) {
    const PrefillArgs &p = a.p;
    CUtensorMap tm[4];
    const void *src[4] = {p.q, p.k, p.v, p.alpha};
    for (int i = 0; i < 4; ++i) {
        std::memset(&tm[i], 0, sizeof(CUtensorMap));
        const uint64_t rows = p.T_tot > 0 ? (uint64_t)p.T_tot : 1;
        if (encode_tmap_bf16_2d(&tm[i], src[i], (uint64_t)p.H * D, rows, (uint64_t)p.H * D * 2, 64, 64) != 0)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)A_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)B_SMEM);
    if (e != cudaSuccess) return e;
    const unsigned chains = (unsigned)(p.nseq * p.H);
    if (plan.nwaves == 0) {   // only empty sequences
        chain_kernel<<<chains, kBThreads, B_SMEM, s>>>(a, 0, 0, 0);
        return cudaGetLastError();
    }
    for (int w = 0; w < plan.nwaves; ++w) {
        const int i0 = plan.wave_begin[w], n = plan.wave_begin[w + 1] - i0;
        if (n > 0) {
            // wave 0: a plain launch; later waves: dependent launches beside the previous chains
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(n * p.H));
            cfg.blockDim = dim3(kAThreads);
            cfg.dynamicSmemBytes = A_SMEM;
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = w > 0 ? 1 : 0;
            e = cudaLaunchKernelEx(&cfg, chunk_prep_kernel, a, w, i0, w > 0 ? 1 : 0, tm[0], tm[1], tm[2], tm[3]);
            if (e != cudaSuccess) return e;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(chains);
        cfg.blockDim = dim3(kBThreads);
        cfg.dynamicSmemBytes = B_SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = n > 0 ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, chain_kernel, a, w, plan.wave_c0[w], plan.wave_c0[w + 1]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda
