// Chunked varlen KDA prefill on the 5th-generation tensor cores (bf16 inputs, d = 128).
//
// What it computes is the token recurrence S_t = (I - beta k k^T) Diag(alpha) S_{t-1} +
// beta k v^T, o_t = S_t^T q_t with the width-4 causal conv on q | k | v ("Lesson 01 ·
// Architecture map", §两种 Attention，两种状态), grouped into chunks of 64 tokens that each act
// on S as one affine map ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제", §0x01 1.3), with
// checkpoints of (S, conv window) streamed at listed chunk ends and the final state written to
// the sequence's active object ("Cache de préfixe hybride KDA–MLA", §Le fonctionnement du
// prefill).
//
// Chunk algebra (rows r, s = 0..63 of one chunk, S = state at the chunk start, gamma_r =
// prod_{u<=r} alpha_u per key channel, gamma_C = gamma_63; padding rows are identity tokens):
//   Kt' = k gamma_r / gamma_C,  Qt' = q gamma_r / gamma_C,  Kb = k gamma_C / gamma_r
//   G = Kt' Kb^T = Kt Kh^T,     P = lower_incl(Qt' Kb^T)          (one M = 128 MMA)
//   T = (I + Diag(beta) strict_lower(G))^{-1} Diag(beta)          (CUDA cores + tf32 mma.sync)
//   WK'^T = Kt'^T T^T,          U^T = V^T T^T                      (two M = 128 MMAs)
//   O^T  = (Gamma_C S)^T Qt'^T  + W^T P^T
//   W^T  = U^T - (Gamma_C S)^T WK'^T
//   S^T <- (Gamma_C S)^T + W^T Kb
// The state lives transposed in TMEM (lane = value channel j, column = key channel i), so every
// state contraction has M = 128; the scaled state (Gamma_C S)^T is also kept in TMEM as the bf16
// A operand of the next contraction.  Decay is anchored at the chunk end, so no per-element
// division is needed.
//
// Warp roles (16 warps): warp 0 issues TMA loads of the raw q, k, v, alpha tiles; warp 1 issues
// all tcgen05.mma from one thread; warps 4-7 ("conv") do the conv and the decay scaling of the
// chunk ahead; warps 8-11 ("solve") do the triangular solve and the WK'^T operand; warps 12-15
// ("seq") run the state epilogues of the current chunk (checkpoint stores, decay of S, W,
// outputs).  The three warpgroups work on three consecutive chunks at once.  Every wait is bounded: on a
// timeout the kernel records KDA_DEV_TIMEOUT, stops issuing work, frees TMEM and returns.
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

constexpr int D = 128;
constexpr int C = kChunk;            // 64
constexpr int kThreads = 512;
constexpr int kPrepWarp0 = 4, kSolveWarp0 = 8, kSeqWarp0 = 12;
constexpr int kBarPrep = 1, kBarSeq = 2, kBarSolve = 3, kBarSolveHalf = 4;

// Shared-memory map (byte offsets from a 1024-aligned base).
constexpr uint32_t OFF_KQ = 0;          // [2 slots][2 kb][128 rows: k 0-63 | q 64-127][128 B]
constexpr uint32_t OFF_KB = 65536;      // [2 slots][2 kb][64 rows][128 B]   Kb
constexpr uint32_t OFF_V = 98304;       // [2 slots][2 kb][64 rows][128 B]   raw v -> V
constexpr uint32_t OFF_AL = 131072;     // [2 slots][2 kb][64 rows][128 B]   raw alpha
constexpr uint32_t OFF_P = 163840;      // [2 slots][64 rows][128 B]         P
constexpr uint32_t OFF_T = 180224;      // [64 rows][128 B]                  T
constexpr uint32_t OFF_WK = 188416;     // [128 rows][128 B] WK'^T; fp32 64x64 solve scratch
constexpr uint32_t OFF_WT = 204800;     // [128 rows][128 B]                 W^T bf16
constexpr uint32_t OFF_GC = 221184;     // float [2][128]                    gamma_C
constexpr uint32_t OFF_BS = 222208;     // float [2][64]                     beta
constexpr uint32_t OFF_RED = 222720;    // float2 [2][64]                    half products of alpha
constexpr uint32_t OFF_HALO = 223744;   // bf16 [3][384]                     conv window
constexpr uint32_t OFF_BAR = 226048;    // mbarriers, flags
constexpr uint32_t OFF_PD = OFF_BAR + 256;   // float [2][64]  exact diagonal of P
constexpr uint32_t SMEM_BYTES = OFF_BAR + 768 + 1024;   // + alignment slack

// TMEM columns.  G|P and WK'^T share columns (their lifetimes do not overlap); the bf16
// operand (Gamma S)^T of M3 lives in the last 64 columns (two values per column).
constexpr uint32_t COL_S = 0, COL_O = 128, COL_W = 256, COL_GP = 384, COL_WK = 384, COL_SA = 448;

// mbarrier indices ([2] arrays indexed by local chunk parity).
enum {
    B_FULL = 0,      // TMA tiles landed             (tx)
    B_P1 = 2,        // prep: operands of the chunk written
    B_GP = 4,        // mma: G|P in TMEM
    B_T = 6,         // prep: T written
    B_M2 = 8,        // mma: WK'^T, U^T done
    B_WK = 10,       // prep: WK'^T operand written
    B_SB = 12,       // seq: (Gamma S)^T operand written, TMEM S scaled
    B_W = 14,        // mma: W^T in TMEM (M3 done)
    B_M3 = 16,       // mma: M3 done (for the solve scratch)
    B_WT = 18,       // seq: W^T operand written, D_W read
    B_M4 = 20,       // mma: chunk done (S advanced, O complete)
    B_DO = 22,       // seq: D_O read
    B_GPF = 24,      // solve: G|P read from TMEM (the next M1 may overwrite it)
    NUM_BARS = 26
};

using namespace tcx;

// ------------------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = ptx::smem_align1024(smem_raw);
    Shared S;
    S.base = sm;
    S.bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    S.err = reinterpret_cast<volatile int *>(sm + OFF_BAR + NUM_BARS * 8);
    S.tmem = reinterpret_cast<uint32_t *>(sm + OFF_BAR + NUM_BARS * 8 + 16);
    volatile int *wg_flag = reinterpret_cast<volatile int *>(sm + OFF_BAR + NUM_BARS * 8 + 32);
    float *gC = reinterpret_cast<float *>(sm + OFF_GC);
    float *bs = reinterpret_cast<float *>(sm + OFF_BS);
    float2 *red = reinterpret_cast<float2 *>(sm + OFF_RED);
    __nv_bfloat16 *halo = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_HALO);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % a.H, sq = blockIdx.x / a.H;
    const SeqMeta m = a.seqs[sq];
    const int H = a.H;
    const uint64_t rec = (uint64_t)h * (uint64_t)a.pool.rec_bytes;
    const int32_t *act_pages = a.pages + m.active_off;
    const int64_t start = m.start_pos, end = m.start_pos + m.len;
    const int64_t c_first = start / C;
    const int nchunks = m.len > 0 ? (int)((end - 1) / C - c_first + 1) : 0;

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) ptx::mbar_init(&S.bar[i], 1);
        *S.err = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(S.tmem, 512);
        ptx::tmem_relinquish();
    }
    // Initial conv window (raw tokens, bf16) from the active object, or zeros.
    for (int e = tid; e < 3 * 3 * D; e += kThreads) {
        __nv_bfloat16 x = __float2bfloat16_rn(0.f);
        if (m.has_init) {
            const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(
                obj_addr(a.pool, act_pages, rec + (uint64_t)D * D * 4 + (uint64_t)e * 2, a.status));
            if (p) x = *p;
        }
        halo[e] = x;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tbase = *S.tmem;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0 && nchunks > 0) {
            ptx::prefetch_tmap(&tm_q);
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_v);
            ptx::prefetch_tmap(&tm_a);
            for (int lc = 0; lc < nchunks && !*S.err; ++lc) {
                const int b = lc & 1;
                if (lc >= 2) {
                    if (!wait_bar(S, B_P1 + b, par(lc - 2))) break;   // alpha slot consumed
                    if (!wait_bar(S, B_M2 + b, par(lc - 2))) break;   // V slot consumed
                    if (!wait_bar(S, B_M4 + b, par(lc - 2))) break;   // KQ slot free
                }
                const int64_t abs0 = (c_first + lc) * C;
                const int32_t y = (int32_t)((int64_t)m.tok_begin + (abs0 - start));
                uint64_t *fb = &S.bar[B_FULL + b];
                ptx::mbar_arrive_expect_tx(fb, 4 * 2 * 64 * 128);
                uint8_t *kq = sm + OFF_KQ + b * 32768;
                for (int kb = 0; kb < 2; ++kb) {
                    const int32_t x = h * D + kb * 64;
                    ptx::tma_load_2d(kq + kb * 16384, &tm_k, fb, x, y);
                    ptx::tma_load_2d(kq + kb * 16384 + 8192, &tm_q, fb, x, y);
                    ptx::tma_load_2d(sm + OFF_V + b * 16384 + kb * 8192, &tm_v, fb, x, y);
                    ptx::tma_load_2d(sm + OFF_AL + b * 16384 + kb * 8192, &tm_a, fb, x, y);
                }
            }
            // Do not leave while copies may still be landing in shared memory.
            if (*S.err)
                for (int lc = 0; lc < nchunks; ++lc) {
                    uint32_t n = 0;
                    while (!ptx::mbar_try_wait(&S.bar[B_FULL + (lc & 1)], par(lc)) && n < ptx::kSpinLimit) ++n;
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && nchunks > 0) {
            const uint32_t id_gp = ptx::idesc_bf16(128, 64, 0, 0);
            const uint32_t id_m2 = ptx::idesc_bf16(128, 64, 1, 0);
            const uint32_t id_o = ptx::idesc_bf16(128, 64, 0, 0);
            const uint32_t id_w = ptx::idesc_bf16(128, 64, 0, 1, 1);
            const uint32_t id_s = ptx::idesc_bf16(128, 128, 0, 1);
            const uint32_t id_op = ptx::idesc_bf16(128, 64, 0, 0);
            const uint32_t sbase = ptx::smem_u32(sm);
            int n1 = 0, n2 = 0, n3 = 0, n4 = 0;
            uint32_t spins = 0;
            while (n4 < nchunks && !*S.err) {
                bool did = false;
                // M3: O^T = SB Qt'^T ; W^T += -SB WK'^T
                if (n3 == n4 && n3 < nchunks) {
                    const int b = n3 & 1;
                    if (ptx::mbar_test(&S.bar[B_SB + b], par(n3)) &&
                        ptx::mbar_test(&S.bar[B_WK + b], par(n3)) &&
                        (n3 < 2 || ptx::mbar_test(&S.bar[B_DO + b], par(n3 - 2)))) {
                        ptx::tc_fence_after();
                        const uint32_t kq = sbase + OFF_KQ + b * 32768, wk = sbase + OFF_WK;
                        for (int s = 0; s < 8; ++s) {
                            const uint64_t bq = ptx::sdesc_sw128(kq + 8192 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                            ptx::mma_bf16_ta(tbase + COL_O + b * 64, tbase + COL_SA + s * 8, bq, id_o, s > 0 ? 1u : 0u);
                        }
                        for (int s = 0; s < 8; ++s) {
                            const uint64_t bw = ptx::sdesc_sw128(wk + s * 2048, 8192, 1024);
                            ptx::mma_bf16_ta(tbase + COL_W + b * 64, tbase + COL_SA + s * 8, bw, id_w, 1u);
                        }
                        ptx::mma_commit(&S.bar[B_W + b]);
                        ptx::mma_commit(&S.bar[B_M3 + b]);
                        ++n3;
                        did = true;
                    }
                }
                // M4: S^T += W^T Kb ; O^T += W^T P^T
                if (n4 < n3) {
                    const int b = n4 & 1;
                    if (ptx::mbar_test(&S.bar[B_WT + b], par(n4))) {
                        ptx::tc_fence_after();
                        const uint32_t wt = sbase + OFF_WT, kb = sbase + OFF_KB + b * 16384, pb = sbase + OFF_P + b * 8192;
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ad = ptx::sdesc_sw128(wt + s * 32, 16, 1024);
                            const uint64_t bd = ptx::sdesc_sw128(kb + s * 2048, 8192, 1024);
                            ptx::mma_bf16(tbase + COL_S, ad, bd, id_s, 1u);
                        }
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ad = ptx::sdesc_sw128(wt + s * 32, 16, 1024);
                            const uint64_t bd = ptx::sdesc_sw128(pb + s * 32, 16, 1024);
                            ptx::mma_bf16(tbase + COL_O + b * 64, ad, bd, id_op, 1u);
                        }
                        ptx::mma_commit(&S.bar[B_M4 + b]);
                        ++n4;
                        did = true;
                    }
                }
                // M1: [Kt'; Qt'] Kb^T -> G | P
                if (n1 < nchunks) {
                    const int b = n1 & 1;
                    if (ptx::mbar_test(&S.bar[B_P1 + b], par(n1)) &&
                        (n1 == 0 || ptx::mbar_test(&S.bar[B_WK + ((n1 - 1) & 1)], par(n1 - 1)))) {
                        ptx::tc_fence_after();
                        const uint32_t kq = sbase + OFF_KQ + b * 32768, kb = sbase + OFF_KB + b * 16384;
                        for (int s = 0; s < 8; ++s) {
                            const uint64_t ad = ptx::sdesc_sw128(kq + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                            const uint64_t bd = ptx::sdesc_sw128(kb + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024);
                            ptx::mma_bf16(tbase + COL_GP, ad, bd, id_gp, s > 0 ? 1u : 0u);
                        }
                        ptx::mma_commit(&S.bar[B_GP + b]);
                        ++n1;
                        did = true;
                    }
                }
                // M2: WK'^T = Kt'^T T^T ; U^T = V^T T^T
                if (n2 < n1) {
                    const int b = n2 & 1;
                    if (ptx::mbar_test(&S.bar[B_T + b], par(n2)) &&
                        (n2 < 2 || ptx::mbar_test(&S.bar[B_WT + b], par(n2 - 2)))) {
                        ptx::tc_fence_after();
                        const uint32_t kq = sbase + OFF_KQ + b * 32768, v = sbase + OFF_V + b * 16384, t = sbase + OFF_T;
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t bd = ptx::sdesc_sw128(t + s * 32, 16, 1024);
                            ptx::mma_bf16(tbase + COL_WK, ptx::sdesc_sw128(kq + s * 2048, 16384, 1024), bd, id_m2,
                                          s > 0 ? 1u : 0u);
                            ptx::mma_bf16(tbase + COL_W + b * 64, ptx::sdesc_sw128(v + s * 2048, 8192, 1024), bd,
                                          id_m2, s > 0 ? 1u : 0u);
                        }
                        ptx::mma_commit(&S.bar[B_M2 + b]);
                        ++n2;
                        did = true;
                    }
                }
                if (did) spins = 0;
                else if (++spins > ptx::kSpinLimit) *S.err = 1;
            }
        }
    } else if (warp >= kPrepWarp0 && warp < kSolveWarp0) {
        // ------------------------------------------------------------------ conv warpgroup
        const int t = tid - kPrepWarp0 * 32;          // 0..127, TMEM lane
        const int p = t & 63, hf = t >> 6;            // channel pair (2p, 2p+1), row half
        const int c0 = 2 * p, kb = c0 >> 6, cb = (c0 & 63) * 2;   // tile block and column byte
        float wq[2][4], wk[2][4], wv[2][4];
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wq[e][j] = a.conv_w[((int64_t)h * 3 * D + c0 + e) * 4 + j];
                wk[e][j] = a.conv_w[((int64_t)h * 3 * D + D + c0 + e) * 4 + j];
                wv[e][j] = a.conv_w[((int64_t)h * 3 * D + 2 * D + c0 + e) * 4 + j];
            }
        const __nv_bfloat16 *betag = static_cast<const __nv_bfloat16 *>(a.beta);
        int nck = 0;   // next checkpoint index of this sequence (window part)
        volatile int *pflag = wg_flag;
        // beta of chunk lc for this thread's row t (t < 64); 0 outside the sequence
        auto load_beta = [&](int lc2) {
            const int64_t a0 = (c_first + lc2) * C;
            const int64_t pos = a0 + t;
            if (pos < start || pos >= end) return 0.f;
            return __bfloat162float(betag[((int64_t)m.tok_begin + (pos - start)) * H + h]);
        };
        float beta_next = (t < C && nchunks > 0) ? load_beta(0) : 0.f;
        for (int lc = 0; lc < nchunks; ++lc) {
            const int b = lc & 1;
            const int64_t abs0 = (c_first + lc) * C;
            const int r_first = start > abs0 ? (int)(start - abs0) : 0;
            const int r_end = end - abs0 < C ? (int)(end - abs0) : C;
            // ---------------- P1: conv, decay, scaled operands
            if (!wg_wait(S, B_FULL + b, par(lc), t, kBarPrep, pflag)) break;
            if (lc >= 2 && !wg_wait(S, B_M4 + b, par(lc - 2), t, kBarPrep, pflag)) break;   // Kb / P slot free
            uint8_t *kq = sm + OFF_KQ + b * 32768;
            uint8_t *kbt = sm + OFF_KB + b * 16384;
            // window carried in from the previous chunk (halo), for both halves
            float2 wqv[3], wkv[3], wvv[3];
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                wqv[u] = make_float2(__bfloat162float(halo[u * 384 + c0]), __bfloat162float(halo[u * 384 + c0 + 1]));
                wkv[u] = make_float2(__bfloat162float(halo[u * 384 + D + c0]), __bfloat162float(halo[u * 384 + D + c0 + 1]));
                wvv[u] = make_float2(__bfloat162float(halo[u * 384 + 2 * D + c0]),
                                     __bfloat162float(halo[u * 384 + 2 * D + c0 + 1]));
            }
            // the second half starts after the last (up to three) valid rows below row 32:
            // shift those raw rows into its window
            if (hf == 1) {
                const int hi = r_end < 32 ? r_end : 32;
                const int lo = (hi - 3) > r_first ? (hi - 3) : r_first;
                for (int r = lo; r < hi; ++r) {
                    const uint32_t off = kb * 16384 + ptx::sw128_off(r, cb);
                    const float2 xq = bf2_to_f2(*reinterpret_cast<const uint32_t *>(kq + off + 8192));
                    const float2 xk = bf2_to_f2(*reinterpret_cast<const uint32_t *>(kq + off));
                    const float2 xv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + OFF_V + b * 16384 + kb * 8192 + ptx::sw128_off(r, cb)));
                    wqv[0] = wqv[1]; wqv[1] = wqv[2]; wqv[2] = xq;
                    wkv[0] = wkv[1]; wkv[1] = wkv[2]; wkv[2] = xk;
                    wvv[0] = wvv[1]; wvv[1] = wvv[2]; wvv[2] = xv;
                }
            }
            // alpha product over this half's rows (four independent partial products)
            float2 ap[4] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f), make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) {
                const int r = hf * 32 + rr;
                const float2 al = bf2_to_f2(*reinterpret_cast<const uint32_t *>(sm + OFF_AL + b * 16384 + kb * 8192 + ptx::sw128_off(r, cb)));
                const bool valid = r >= r_first && r < r_end;
                ap[rr & 3].x *= valid ? al.x : 1.f;
                ap[rr & 3].y *= valid ? al.y : 1.f;
            }
            red[hf * 64 + p] = make_float2((ap[0].x * ap[1].x) * (ap[2].x * ap[3].x), (ap[0].y * ap[1].y) * (ap[2].y * ap[3].y));
            if (t < C) bs[b * 64 + t] = beta_next;
            named_bar(kBarPrep, 128);
            // fetch the next chunk's beta now; it is needed only one chunk later
            if (t < C && lc + 1 < nchunks) beta_next = load_beta(lc + 1);
            const float2 h0 = red[p], h1 = red[64 + p];
            const float gCx = h0.x * h1.x, gCy = h0.y * h1.y;
            const float icx = 1.f / gCx, icy = 1.f / gCy;
            if (hf == 0) {
                gC[b * 128 + c0] = gCx;
                gC[b * 128 + c0 + 1] = gCy;
                if (!(gCx >= kMinChunkDecay && gCy >= kMinChunkDecay)) flag_status(a.status, KDA_DEV_RANGE);
            }
            float gx = hf ? h0.x : 1.f, gy = hf ? h0.y : 1.f;
            // One row: conv of q | k | v, running decay, scaled bf16 operands written in place
            // (q, k, v tiles) and to Kb; rows outside the sequence become zeros.  The 128-byte
            // swizzle of a row depends only on r mod 8, so the eight in-row offsets of this
            // thread's channel pair are computed once; full chunks take a branch-free path of
            // eight rows at a time with all loads issued before the in-place stores.
            uint32_t swz[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) swz[u] = ptx::sw128_off(u, cb);
            uint8_t *const qrow = kq + kb * 16384 + 8192, *const krow = kq + kb * 16384;
            uint8_t *const vrow = sm + OFF_V + b * 16384 + kb * 8192, *const arow = sm + OFF_AL + b * 16384 + kb * 8192;
            uint8_t *const kbrow = kbt + kb * 8192;
            auto row_proc = [&](uint32_t off, float2 xq, float2 xk, float2 xv, float2 al, bool valid) {
                uint32_t oq = 0, ok = 0, okb = 0, ov = 0;
                float dpart = 0.f;
                if (valid) {
                    const float qb0 = wq[0][0] * wqv[0].x + wq[0][1] * wqv[1].x + wq[0][2] * wqv[2].x + wq[0][3] * xq.x;
                    const float qb1 = wq[1][0] * wqv[0].y + wq[1][1] * wqv[1].y + wq[1][2] * wqv[2].y + wq[1][3] * xq.y;
                    const float kb0 = wk[0][0] * wkv[0].x + wk[0][1] * wkv[1].x + wk[0][2] * wkv[2].x + wk[0][3] * xk.x;
                    const float kb1 = wk[1][0] * wkv[0].y + wk[1][1] * wkv[1].y + wk[1][2] * wkv[2].y + wk[1][3] * xk.y;
                    const float vb0 = wv[0][0] * wvv[0].x + wv[0][1] * wvv[1].x + wv[0][2] * wvv[2].x + wv[0][3] * xv.x;
                    const float vb1 = wv[1][0] * wvv[0].y + wv[1][1] * wvv[1].y + wv[1][2] * wvv[2].y + wv[1][3] * xv.y;
                    wqv[0] = wqv[1]; wqv[1] = wqv[2]; wqv[2] = xq;
                    wkv[0] = wkv[1]; wkv[1] = wkv[2]; wkv[2] = xk;
                    wvv[0] = wvv[1]; wvv[1] = wvv[2]; wvv[2] = xv;
                    gx *= al.x;
                    gy *= al.y;
                    // this pair's share of the diagonal P[r][r] = qbar_r . kbar_r (the decay cancels)
                    dpart = qb0 * kb0 + qb1 * kb1;
                    const float sx = gx * icx, sy = gy * icy;      // gamma_r / gamma_C
                    oq = pack_bf16x2(qb0 * sx, qb1 * sy);
                    ok = pack_bf16x2(kb0 * sx, kb1 * sy);
                    okb = pack_bf16x2(kb0 * rcp_approx(sx), kb1 * rcp_approx(sy));
                    ov = pack_bf16x2(vb0, vb1);
                }
                *reinterpret_cast<float *>(arow + off) = dpart;   // alpha slot, already read
                *reinterpret_cast<uint32_t *>(qrow + off) = oq;
                *reinterpret_cast<uint32_t *>(krow + off) = ok;
                *reinterpret_cast<uint32_t *>(kbrow + off) = okb;
                *reinterpret_cast<uint32_t *>(vrow + off) = ov;
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
                            row_proc((uint32_t)(r0 + h4 + u) * 128u + (swz[h4 + u] & 127u), xq[u], xk[u], xv[u],
                                     al[u], true);
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
                    row_proc(off, xq, xk, xv, al, r >= r_first && r < r_end);
                }
            }
            named_bar(kBarPrep, 128);
            if (t < C) {
                float acc = 0.f;
                for (int pp = 0; pp < 64; ++pp)
                    acc += *reinterpret_cast<const float *>(sm + OFF_AL + b * 16384 + (pp >> 5) * 8192 +
                                                            ptx::sw128_off(t, (pp & 31) * 4));
                reinterpret_cast<float *>(sm + OFF_PD)[b * 64 + t] = acc;
            }
            ptx::fence_proxy_async_smem();
            named_bar(kBarPrep, 128);
            if (t == 0) ptx::mbar_arrive(&S.bar[B_P1 + b]);
            // conv window after this chunk (second half holds it): keep for the next chunk and
            // store it into a checkpoint that ends here, or into the active object at the end.
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
            named_bar(kBarPrep, 128);
            {
                const int64_t cend = abs0 + r_end;
                while (nck < m.ckpt_count) {
                    const CkptMeta ck = a.ckpts[m.ckpt_begin + nck];
                    if (ck.pos > cend) break;
                    if (ck.pos == cend) {
                        const int32_t *pg = a.pages + ck.pages_off;
                        for (int e = t; e < 9 * D; e += 128) {
                            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(
                                obj_addr(a.pool, pg, rec + (uint64_t)D * D * 4 + (uint64_t)e * 2, a.status));
                            if (dst) *dst = halo[e];
                        }
                    }
                    ++nck;
                }
            }
        }
        // final conv window into the active object
        for (int e = t; e < 9 * D; e += 128) {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(
                obj_addr(a.pool, act_pages, rec + (uint64_t)D * D * 4 + (uint64_t)e * 2, a.status));
            if (dst) *dst = halo[e];
        }
    } else if (warp >= kSolveWarp0 && warp < kSeqWarp0) {
        // ------------------------------------------------------------------ solve warpgroup
        // T of chunk lc (G | P from TMEM, triangular solve) and the WK'^T operand, while the conv
        // warpgroup already prepares chunk lc + 1.
        const int t = tid - kSolveWarp0 * 32;         // 0..127, TMEM lane
        float *Msc = reinterpret_cast<float *>(sm + OFF_WK);
        volatile int *pflag = wg_flag + 2;
        for (int lc = 0; lc < nchunks; ++lc) {
            const int b = lc & 1;
            // ---------------- P2: G | P from TMEM, T = (I + A)^{-1} Diag(beta)
            if (!wg_wait(S, B_GP + b, par(lc), t, kBarSolve, pflag)) break;
            if (!wg_wait(S, B_P1 + b, par(lc), t, kBarSolve, pflag)) break;              // beta, diag of P
            if (lc >= 1 && !wg_wait(S, B_M3 + ((lc - 1) & 1), par(lc - 1), t, kBarSolve, pflag)) break;   // scratch free
            if (lc >= 2 && !wg_wait(S, B_M4 + b, par(lc - 2), t, kBarSolve, pflag)) break;   // P slot free
            ptx::tc_fence_after();
            {
                float g0[32], g1[32];
                const uint32_t ta = tbase + ((uint32_t)((warp - kSolveWarp0) * 32) << 16) + COL_GP;
                ptx::tmem_ld32(ta, g0);
                ptx::tmem_ld32(ta + 32, g1);
                ptx::tmem_wait_ld();
                if (t < C) {
                    // A row r = beta_r * strict_lower(G) (fp32 scratch, swizzled float4 groups)
                    const int r = t;
                    const float br = bs[b * 64 + r];
                    float4 *row = reinterpret_cast<float4 *>(Msc + r * 64);
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        float e[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int s2 = c4 * 4 + u;
                            const float gv = s2 < 32 ? g0[s2 & 31] : g1[s2 & 31];
                            e[u] = s2 < r ? br * gv : 0.f;
                        }
                        row[c4 ^ (r & 7)] = make_float4(e[0], e[1], e[2], e[3]);
                    }
                } else {
                    // P row r = lower_incl(Qt' Kb^T), with the exact fp32 diagonal
                    const int r = t - C;
                    uint8_t *pr = sm + OFF_P + b * 8192;
                    const float pd = reinterpret_cast<const float *>(sm + OFF_PD)[b * 64 + r];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 v;
                        uint32_t *vv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const int s0 = ch * 8 + q2 * 2;
                            const float ga = s0 < 32 ? g0[s0 & 31] : g1[s0 & 31];
                            const float gb = s0 + 1 < 32 ? g0[(s0 + 1) & 31] : g1[(s0 + 1) & 31];
                            vv[q2] = pack_bf16x2(s0 < r ? ga : (s0 == r ? pd : 0.f),
                                                 s0 + 1 < r ? gb : (s0 + 1 == r ? pd : 0.f));
                        }
                        *reinterpret_cast<uint4 *>(pr + ptx::sw128_off(r, ch * 16)) = v;
                    }
                }
            }
            ptx::tc_fence_before();
            named_bar(kBarSolve, 128);
            // level 0: invert the four 16x16 diagonal blocks, one row per thread.  Row x of the
            // inverse solves x (I + A_bb) = e_r; eliminating from the last row upward needs only
            // rows of A_bb, which every thread of the block reads (broadcast), and no predicate:
            // x[m] is still zero for m above the thread's own row.
            if (t < C) {
                const int r = t, bb = r >> 4, rr = r & 15;
                float x[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) x[c] = c == rr ? 1.f : 0.f;
#pragma unroll
                for (int mm = 15; mm >= 1; --mm) {
                    const int ar = bb * 16 + mm;
                    const float4 *arow = reinterpret_cast<const float4 *>(Msc + ar * 64);
                    float av[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (q * 4 < mm) {
                            const float4 v4 = arow[(bb * 4 + q) ^ (ar & 7)];
                            av[q * 4] = v4.x; av[q * 4 + 1] = v4.y; av[q * 4 + 2] = v4.z; av[q * 4 + 3] = v4.w;
                        }
                    }
                    const float xm = x[mm];
#pragma unroll
                    for (int c = 0; c < mm; ++c) x[c] = fmaf(-xm, av[c], x[c]);
                }
                named_bar(kBarSolveHalf, 64);
                float4 *row = reinterpret_cast<float4 *>(Msc + r * 64);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    row[(bb * 4 + q) ^ (r & 7)] = make_float4(x[q * 4], x[q * 4 + 1], x[q * 4 + 2], x[q * 4 + 3]);
            }
            named_bar(kBarSolve, 128);
            // Off-diagonal blocks of Inv = (I + A)^{-1}, in 32 x 32 halves (tf32 mma.sync, one
            // warp per 16 x 16 block).  With J0, J1 the inverses of the two diagonal 32 x 32 blocks
            // and B the lower-left 32 x 32 block of A:
            //   J0 = [[I00, 0], [-I11 A10 I00, I11]],  J1 likewise from blocks 2, 3,
            //   lower-left of Inv = -J1 (B J0).
            {
                const int pw = warp - kSolveWarp0;
                const float zero4[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                // step A: X10 = -I11 (A10 I00) on warp 0, X32 = -I33 (A32 I22) on warp 1
                if (pw < 2) {
                    const int i = pw == 0 ? 1 : 3, j = i - 1;
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    blk_mma(acc, Msc, i, j, j, lane);
                    __syncwarp();
                    blk_store(Msc, i, j, acc, 1.f, lane);
                    __syncwarp();
                    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    blk_mma(acc2, Msc, i, i, j, lane);
                    __syncwarp();
                    blk_store(Msc, i, j, acc2, -1.f, lane);
                }
                named_bar(kBarSolve, 128);
                // step B1: Y = B J0, block (bi, bj) = (2 + pw / 2, pw % 2) per warp
                const int bi = 2 + (pw >> 1), bj = pw & 1;
                float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if (bj == 0) {
                    blk_mma(y, Msc, bi, 0, 0, lane);     // A_i0 I00
                    blk_mma(y, Msc, bi, 1, 0, lane);     // A_i1 X10
                } else {
                    blk_mma(y, Msc, bi, 1, 1, lane);     // A_i1 I11
                }
                named_bar(kBarSolve, 128);
                blk_store(Msc, bi, bj, y, 1.f, lane);
                named_bar(kBarSolve, 128);
                // step B2: Z = -J1 Y
                float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if (bi == 2) {
                    blk_mma(z, Msc, 2, 2, bj, lane);     // I22 Y2j
                } else {
                    blk_mma(z, Msc, 3, 2, bj, lane);     // X32 Y2j
                    blk_mma(z, Msc, 3, 3, bj, lane);     // I33 Y3j
                }
                named_bar(kBarSolve, 128);
                blk_store(Msc, bi, bj, z, -1.f, lane);
                (void)zero4;
            }
            named_bar(kBarSolve, 128);
            // T = Inv Diag(beta) -> bf16 operand [r][s]
            if (t < C) {
                const int r = t;
                const float4 *row = reinterpret_cast<const float4 *>(Msc + r * 64);
                const float4 *b4 = reinterpret_cast<const float4 *>(bs + b * 64);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float e[8];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int c4 = ch * 2 + h2;
                        const float4 mv = row[c4 ^ (r & 7)];
                        const float4 bv = b4[c4];
                        e[h2 * 4 + 0] = c4 * 4 + 0 <= r ? mv.x * bv.x : 0.f;
                        e[h2 * 4 + 1] = c4 * 4 + 1 <= r ? mv.y * bv.y : 0.f;
                        e[h2 * 4 + 2] = c4 * 4 + 2 <= r ? mv.z * bv.z : 0.f;
                        e[h2 * 4 + 3] = c4 * 4 + 3 <= r ? mv.w * bv.w : 0.f;
                    }
                    uint4 v;
                    v.x = pack_bf16x2(e[0], e[1]);
                    v.y = pack_bf16x2(e[2], e[3]);
                    v.z = pack_bf16x2(e[4], e[5]);
                    v.w = pack_bf16x2(e[6], e[7]);
                    *reinterpret_cast<uint4 *>(sm + OFF_T + ptx::sw128_off(r, ch * 16)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
            named_bar(kBarSolve, 128);
            if (t == 0) ptx::mbar_arrive(&S.bar[B_T + b]);
            // ---------------- P3: WK'^T from TMEM -> bf16 operand rows (row = key channel)
            if (!wg_wait(S, B_M2 + b, par(lc), t, kBarSolve, pflag)) break;
            ptx::tc_fence_after();
            {
                float w0[32], w1[32];
                const uint32_t ta = tbase + ((uint32_t)((warp - kSolveWarp0) * 32) << 16) + COL_WK;
                ptx::tmem_ld32(ta, w0);
                ptx::tmem_ld32(ta + 32, w1);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 v;
                    uint32_t *vv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int c = ch * 8 + 2 * q2;
                        vv[q2] = c < 32 ? pack_bf16x2(w0[c & 31], w0[(c + 1) & 31])
                                        : pack_bf16x2(w1[c & 31], w1[(c + 1) & 31]);
                    }
                    *reinterpret_cast<uint4 *>(sm + OFF_WK + ptx::sw128_off(t, ch * 16)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            named_bar(kBarSolve, 128);
            if (t == 0) ptx::mbar_arrive(&S.bar[B_WK + b]);
        }
    } else if (warp >= kSeqWarp0) {
        // ------------------------------------------------------------------ seq warpgroup
        const int j = tid - kSeqWarp0 * 32;           // value channel = TMEM lane
        const uint32_t lanes = (uint32_t)((warp - kSeqWarp0) * 32) << 16;
        __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(a.o);
        // initial state (S^T row j = column j of S)
        for (int i0 = 0; i0 < D; i0 += 32) {
            float v[32];
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                float x = 0.f;
                if (m.has_init) {
                    const float *p = reinterpret_cast<const float *>(
                        obj_addr(a.pool, act_pages, rec + ((uint64_t)(i0 + ii) * D + j) * 4, a.status));
                    if (p) x = *p;
                }
                v[ii] = x;
            }
            ptx::tmem_st32(tbase + lanes + COL_S + i0, v);
        }
        ptx::tmem_wait_st();
        int nck = 0;
        auto write_state_ckpts = [&](int64_t cend, bool final_state) {
            // S (fp32, from TMEM) into the checkpoints ending at cend, and the active object
            bool any = final_state;
            int k = nck;
            while (k < m.ckpt_count && a.ckpts[m.ckpt_begin + k].pos <= cend) {
                if (a.ckpts[m.ckpt_begin + k].pos == cend) any = true;
                ++k;
            }
            if (!any) {
                nck = k;
                return;
            }
            for (int i0 = 0; i0 < D; i0 += 32) {
                float v[32];
                ptx::tmem_ld32(tbase + lanes + COL_S + i0, v);
                ptx::tmem_wait_ld();
                for (int kk = nck; kk < k; ++kk) {
                    const CkptMeta ck = a.ckpts[m.ckpt_begin + kk];
                    if (ck.pos != cend) continue;
                    const int32_t *pg = a.pages + ck.pages_off;
#pragma unroll 4
                    for (int ii = 0; ii < 32; ++ii) {
                        float *dst = reinterpret_cast<float *>(
                            obj_addr(a.pool, pg, rec + ((uint64_t)(i0 + ii) * D + j) * 4, a.status));
                        if (dst) *dst = v[ii];
                    }
                }
                if (final_state) {
#pragma unroll 4
                    for (int ii = 0; ii < 32; ++ii) {
                        float *dst = reinterpret_cast<float *>(
                            obj_addr(a.pool, act_pages, rec + ((uint64_t)(i0 + ii) * D + j) * 4, a.status));
                        if (dst) *dst = v[ii];
                    }
                }
            }
            nck = k;
        };
        auto store_outputs = [&](int lc) {
            const int b = lc & 1;
            const int64_t abs0 = (c_first + lc) * C;
            const int r_first = start > abs0 ? (int)(start - abs0) : 0;
            const int r_end = end - abs0 < C ? (int)(end - abs0) : C;
            const int64_t row0 = (int64_t)m.tok_begin + (abs0 - start);
            for (int r0 = 0; r0 < C; r0 += 32) {
                float v[32];
                ptx::tmem_ld32(tbase + lanes + COL_O + b * 64 + r0, v);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int rr = 0; rr < 32; ++rr) {
                    const int r = r0 + rr;
                    if (r >= r_first && r < r_end) og[((row0 + r) * H + h) * D + j] = __float2bfloat16_rn(v[rr]);
                }
            }
            ptx::tc_fence_before();
            named_bar(kBarSeq, 128);
            if (j == 0) ptx::mbar_arrive(&S.bar[B_DO + b]);
        };
        volatile int *sflag = wg_flag + 1;
        bool ok = true;
        for (int lc = 0; lc < nchunks; ++lc) {
            const int b = lc & 1;
            // ---------------- E1: checkpoint S, decay S by gamma_C in TMEM, bf16 operand
            if (lc >= 1) {
                if (!(ok = wg_wait(S, B_M4 + ((lc - 1) & 1), par(lc - 1), j, kBarSeq, sflag))) break;
                ptx::tc_fence_after();
                write_state_ckpts((c_first + lc) * C, false);
            }
            if (!(ok = wg_wait(S, B_P1 + b, par(lc), j, kBarSeq, sflag))) break;
            const float *gcb = gC + b * 128;
            for (int i0 = 0; i0 < D; i0 += 64) {
                float v[32], w[32], pk[32];
                ptx::tmem_ld32(tbase + lanes + COL_S + i0, v);
                ptx::tmem_ld32(tbase + lanes + COL_S + i0 + 32, w);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    v[ii] *= gcb[i0 + ii];
                    w[ii] *= gcb[i0 + 32 + ii];
                }
                ptx::tmem_st32(tbase + lanes + COL_S + i0, v);
                ptx::tmem_st32(tbase + lanes + COL_S + i0 + 32, w);
                // bf16 row j of (Gamma S)^T, two values per TMEM column: columns i0/2 .. i0/2 + 31
#pragma unroll
                for (int q2 = 0; q2 < 16; ++q2) {
                    pk[q2] = __uint_as_float(pack_bf16x2(v[2 * q2], v[2 * q2 + 1]));
                    pk[16 + q2] = __uint_as_float(pack_bf16x2(w[2 * q2], w[2 * q2 + 1]));
                }
                ptx::tmem_st32(tbase + lanes + COL_SA + (i0 >> 1), pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            named_bar(kBarSeq, 128);
            if (j == 0) ptx::mbar_arrive(&S.bar[B_SB + b]);
            // ---------------- E3 of the previous chunk (off the critical path)
            if (lc >= 1) store_outputs(lc - 1);
            // ---------------- E2: W^T -> bf16 operand
            if (!(ok = wg_wait(S, B_W + b, par(lc), j, kBarSeq, sflag))) break;
            ptx::tc_fence_after();
            for (int r0 = 0; r0 < C; r0 += 32) {
                float v[32];
                ptx::tmem_ld32(tbase + lanes + COL_W + b * 64 + r0, v);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint4 pk;
                    uint32_t *pp = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) pp[q2] = pack_bf16x2(v[ch * 8 + 2 * q2], v[ch * 8 + 2 * q2 + 1]);
                    *reinterpret_cast<uint4 *>(sm + OFF_WT + ptx::sw128_off(j, r0 * 2 + ch * 16)) = pk;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            named_bar(kBarSeq, 128);
            if (j == 0) ptx::mbar_arrive(&S.bar[B_WT + b]);
        }
        if (nchunks > 0 && ok && wg_wait(S, B_M4 + ((nchunks - 1) & 1), par(nchunks - 1), j, kBarSeq, sflag)) {
            ptx::tc_fence_after();
            write_state_ckpts(end, true);
            store_outputs(nchunks - 1);
        } else if (nchunks == 0) {
            write_state_ckpts(end, true);
        }
    }
    // ---------------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (*S.err && tid == 0) flag_status(a.status, KDA_DEV_TIMEOUT);
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tbase, 512);
    }
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) { return a.dtype == KDA_BF16 && a.d == 128; }

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    const int64_t T_tot = a.T_tot;
    CUtensorMap tm[4];
    const void *src[4] = {a.q, a.k, a.v, a.alpha};
    for (int i = 0; i < 4; ++i) {
        std::memset(&tm[i], 0, sizeof(CUtensorMap));
        const uint64_t rows = T_tot > 0 ? (uint64_t)T_tot : 1;
        if (encode_tmap_bf16_2d(&tm[i], src[i], (uint64_t)a.H * D, rows, (uint64_t)a.H * D * 2, 64, 64) != 0)
            return cudaErrorInvalidValue;
    }
    auto kern = prefill_tc_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(a.nseq * a.H), kThreads, SMEM_BYTES, s>>>(a, tm[0], tm[1], tm[2], tm[3]);
    return cudaGetLastError();
}

}  // namespace kda
