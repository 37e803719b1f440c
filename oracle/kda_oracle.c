/*
 * KDA oracle: plain fp64 CPU implementation of the Kimi Delta Attention state path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU-baseline
 * leg of bench.py may load this code.  It shares nothing with the CUDA library
 * (no headers, no helpers, no tables) and the CUDA library never calls it.
 *
 * What it computes, per (sequence, head), token by token, in the order the sources give:
 *
 *   1. Short causal depthwise convolution over the q|k|v channels (width 4, no bias, no
 *      activation).  Tap j of channel c multiplies the raw value of token t-3+j, so tap 3
 *      is the current token.  Tokens before the start come from the conv window (the last
 *      three raw tokens), which is zero for a fresh sequence.
 *      Source: "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" (KDA's AI-infrastructure
 *      challenges), §0x01 (KDA keeps a convolution state of recent tokens) and §0x08 8.2.3
 *      (prefill applies a causal conv to each of q, k, v).
 *   2. Recurrent update with decay first, then the delta-rule write, then the read:
 *        S  <- Diag(alpha_t) S                 (row i = key channel i)
 *        w  =  beta_t (v_t - S^T k_t)
 *        S  <- S + k_t w^T
 *        o_t = S^T q_t
 *      which is S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T.
 *      Source: "Lesson 01 · Architecture map", §"两种 Attention，两种状态" item 1 (the
 *      prose order: decay with the channel-wise forget gate, write with the delta rule,
 *      read with q).  The printed formula on that page leaves S_{t-1} undecayed; the prose
 *      order is the reading adopted here.
 *   3. Checkpoint emission: after the tokens [0, p) of a sequence have been consumed, the
 *      state S and the conv window (raw tokens p-3, p-2, p-1) are copied out.
 *      Source: "Cache de préfixe hybride KDA–MLA", §"Le fonctionnement du prefill".
 *
 * It also builds the affine map of a token segment explicitly,
 *      F_C(S) = M_C S + b_C,  M_t = (I - beta k k^T) Diag(alpha),  b_t = beta k v^T,
 * by multiplying the per-token maps in order (M <- M_t M, b <- M_t b + b_t).
 * Source: KDA's AI-infrastructure challenges, §0x01 1.3 (segment map and its composition)
 * and §0x09 9.1 (closed form S_n = M_n..M_1 S_0 + sum_i M_n..M_{i+1} b_i).
 *
 * Layouts (all fp64, contiguous):
 *   q, k, v, alpha : [T_tot][H][d]        beta : [T_tot][H]
 *   conv_w         : [H][3d][4]           (channel order q | k | v)
 *   S              : [d][d]               (S[i][j], i = key channel, j = value channel)
 *   window         : [3][3d]              (oldest raw token first)
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Plain recurrence on post-conv values for one (sequence, head).
 * kb, vb, qb, al: [T][ld] with the d values of token t at row t; be: [T] with stride be_ld.
 * S: in/out [d][d].  o: [T][o_ld] or NULL. */
static void scan_one(int64_t T, int32_t d,
                     const double *qb, const double *kb, const double *vb, int64_t ld,
                     const double *al, int64_t al_ld, const double *be, int64_t be_ld,
                     double *S, double *o, int64_t o_ld, double *w)
{
    for (int64_t t = 0; t < T; ++t) {
        const double *kt = kb + t * ld, *vt = vb + t * ld, *qt = qb + t * ld;
        const double *at = al + t * al_ld;
        const double bt = be[t * be_ld];
        /* decay: row i scaled by alpha_t[i] */
        for (int32_t i = 0; i < d; ++i)
            for (int32_t j = 0; j < d; ++j)
                S[(int64_t)i * d + j] *= at[i];
        /* delta-rule write vector w = beta (v - S^T k) */
        for (int32_t j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i)
                acc += S[(int64_t)i * d + j] * kt[i];
            w[j] = bt * (vt[j] - acc);
        }
        /* S <- S + k w^T */
        for (int32_t i = 0; i < d; ++i)
            for (int32_t j = 0; j < d; ++j)
                S[(int64_t)i * d + j] += kt[i] * w[j];
        /* read o = S^T q */
        if (o) {
            for (int32_t j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int32_t i = 0; i < d; ++i)
                    acc += S[(int64_t)i * d + j] * qt[i];
                o[t * o_ld + j] = acc;
            }
        }
    }
}

/* Recurrence alone on post-conv inputs of one (sequence, head); all arrays [T][d], beta [T].
 * S is in/out [d][d]; o may be NULL. */
int oracle_scan(int64_t T, int32_t d, const double *qbar, const double *kbar, const double *vbar,
                const double *alpha, const double *beta, double *S, double *o)
{
    if (T < 0 || d <= 0) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)d);
    if (!w) return -2;
    scan_one(T, d, qbar, kbar, vbar, d, alpha, d, beta, 1, S, o, d, w);
    free(w);
    return 0;
}

/* Explicit affine map of a segment of T tokens (post-conv inputs): M [d][d], b [d][d]. */
int oracle_segment_affine(int64_t T, int32_t d, const double *kbar, const double *vbar,
                          const double *alpha, const double *beta, double *M, double *b)
{
    if (T < 0 || d <= 0) return -1;
    const size_t dd = (size_t)d * (size_t)d;
    double *Mt = (double *)malloc(sizeof(double) * dd);
    double *tmp = (double *)malloc(sizeof(double) * dd);
    if (!Mt || !tmp) { free(Mt); free(tmp); return -2; }
    for (size_t x = 0; x < dd; ++x) { M[x] = 0.0; b[x] = 0.0; }
    for (int32_t i = 0; i < d; ++i) M[(size_t)i * d + i] = 1.0;
    for (int64_t t = 0; t < T; ++t) {
        const double *kt = kbar + t * d, *vt = vbar + t * d, *at = alpha + t * d;
        const double bt = beta[t];
        /* M_t = (I - beta k k^T) Diag(alpha) : M_t[i][m] = (delta_im - beta k_i k_m) alpha_m */
        for (int32_t i = 0; i < d; ++i)
            for (int32_t m = 0; m < d; ++m)
                Mt[(size_t)i * d + m] = ((i == m ? 1.0 : 0.0) - bt * kt[i] * kt[m]) * at[m];
        /* M <- M_t M */
        for (int32_t i = 0; i < d; ++i)
            for (int32_t j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int32_t m = 0; m < d; ++m) acc += Mt[(size_t)i * d + m] * M[(size_t)m * d + j];
                tmp[(size_t)i * d + j] = acc;
            }
        memcpy(M, tmp, sizeof(double) * dd);
        /* b <- M_t b + beta k v^T */
        for (int32_t i = 0; i < d; ++i)
            for (int32_t j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int32_t m = 0; m < d; ++m) acc += Mt[(size_t)i * d + m] * b[(size_t)m * d + j];
                tmp[(size_t)i * d + j] = acc + bt * kt[i] * vt[j];
            }
        memcpy(b, tmp, sizeof(double) * dd);
    }
    free(Mt);
    free(tmp);
    return 0;
}

/*
 * Full path for a packed varlen batch: conv + recurrence + checkpoint emission.
 *   cu_seqlens [nseq+1]     token offsets into the packed arrays
 *   S0  [nseq][H][d][d]     initial states (NULL = zeros)
 *   win0[nseq][H][3][3d]    initial conv windows (NULL = zeros)
 *   o   [T_tot][H][d]       outputs
 *   S_out, win_out          final states / windows (same layouts as S0 / win0; may be NULL)
 *   xbar [T_tot][H][3d]     post-conv q|k|v (may be NULL)
 *   ck_off [nseq+1], ck_at[]: for sequence s, entries ck_at[ck_off[s] .. ck_off[s+1]) are
 *                           token counts p (1..len, ascending) after which (S, window) is
 *                           copied to ck_S [n][H][d][d] and ck_win [n][H][3][3d].
 * Threads run over the independent (sequence, head) pairs.
 */
int oracle_kda_run(int32_t nseq, const int64_t *cu_seqlens, int32_t H, int32_t d,
                   const double *q, const double *k, const double *v,
                   const double *alpha, const double *beta, const double *conv_w,
                   const double *S0, const double *win0,
                   double *o, double *S_out, double *win_out, double *xbar,
                   const int64_t *ck_off, const int64_t *ck_at, double *ck_S, double *ck_win)
{
    if (nseq < 0 || H <= 0 || d <= 0) return -1;
    const int32_t C = 3 * d;
    const int64_t npairs = (int64_t)nseq * H;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pair = 0; pair < npairs; ++pair) {
        const int32_t s = (int32_t)(pair / H), h = (int32_t)(pair % H);
        const int64_t t0 = cu_seqlens[s], T = cu_seqlens[s + 1] - cu_seqlens[s];
        double *S = (double *)calloc((size_t)d * d, sizeof(double));
        double *win = (double *)calloc((size_t)3 * C, sizeof(double));
        double *xr = (double *)malloc(sizeof(double) * (size_t)C);
        double *xc = (double *)malloc(sizeof(double) * (size_t)C);
        double *w = (double *)malloc(sizeof(double) * (size_t)d);
        if (!S || !win || !xr || !xc || !w) {
#pragma omp atomic write
            err = -2;
            free(S); free(win); free(xr); free(xc); free(w);
            continue;
        }
        if (S0) memcpy(S, S0 + ((int64_t)s * H + h) * d * d, sizeof(double) * (size_t)d * d);
        if (win0) memcpy(win, win0 + ((int64_t)s * H + h) * 3 * C, sizeof(double) * 3 * (size_t)C);
        const double *wc = conv_w + (int64_t)h * C * 4;
        int64_t ck = ck_off ? ck_off[s] : 0;
        const int64_t ck_end = ck_off ? ck_off[s + 1] : 0;
        for (int64_t t = 0; t < T; ++t) {
            const int64_t row = (t0 + t) * H + h;
            for (int32_t c = 0; c < d; ++c) {
                xr[c] = q[row * d + c];
                xr[d + c] = k[row * d + c];
                xr[2 * d + c] = v[row * d + c];
            }
            /* causal depthwise conv: tap j multiplies raw token t-3+j */
            for (int32_t c = 0; c < C; ++c) {
                const double *wk = wc + (int64_t)c * 4;
                xc[c] = wk[0] * win[c] + wk[1] * win[C + c] + wk[2] * win[2 * C + c] + wk[3] * xr[c];
            }
            /* shift the window: drop the oldest, append the current raw token */
            memmove(win, win + C, sizeof(double) * 2 * (size_t)C);
            memcpy(win + 2 * C, xr, sizeof(double) * (size_t)C);
            if (xbar) memcpy(xbar + row * C, xc, sizeof(double) * (size_t)C);
            /* one recurrence step on the post-conv values */
            scan_one(1, d, xc, xc + d, xc + 2 * d, 0, alpha + row * d, 0, beta + row, 0,
                     S, o + row * d, 0, w);
            /* checkpoint after t+1 tokens */
            while (ck < ck_end && ck_at[ck] == t + 1) {
                memcpy(ck_S + (ck * H + h) * d * d, S, sizeof(double) * (size_t)d * d);
                memcpy(ck_win + (ck * H + h) * 3 * C, win, sizeof(double) * 3 * (size_t)C);
                ++ck;
            }
        }
        if (S_out) memcpy(S_out + ((int64_t)s * H + h) * d * d, S, sizeof(double) * (size_t)d * d);
        if (win_out) memcpy(win_out + ((int64_t)s * H + h) * 3 * C, win, sizeof(double) * 3 * (size_t)C);
        free(S); free(win); free(xr); free(xc); free(w);
    }
    return err;
}

/* Number of threads the parallel region uses (reported with CPU timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
