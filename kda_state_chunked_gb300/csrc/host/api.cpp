// C ABI of libkda.so: argument validation, checkpoint planning, metadata upload and kernel
// launches.  Every GPU call is stream-ordered and makes no host synchronisation except
// when a pinned staging slot is still in use by an earlier copy.
#include <algorithm>
#include <cstring>
#include <vector>

#include "kda.h"
#include "pool.h"
#include "split_plan.h"
#include "../kda_internal.h"

namespace {

using kda::CkptMeta;
using kda::make_split_plan;
using kda::SeqMeta;
using kda::split_applies;

bool valid_shape(int32_t H, int32_t d, int32_t dtype) {
    return H > 0 && H <= 4096 && (d == 64 || d == 128) && (dtype == KDA_F32 || dtype == KDA_BF16);
}

int64_t elem_size(int32_t dtype) { return dtype == KDA_BF16 ? 2 : 4; }

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Pages written by a call must be private to it: allocated, refcount exactly 1, and not
// repeated (a checkpoint visible to others is never written in place).  `g` is the
// duplicate-check generation of this call (kda::pool_new_stamp).
int check_private(kda_pool *p, const int32_t *ids, int64_t n, uint32_t g) {
    for (int64_t i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (id < 0 || id >= p->num_pages) return KDA_EINVAL;
        if (p->ref[id] != 1 || p->stamp[id] == g) return KDA_EREF;
        p->stamp[id] = g;
    }
    return KDA_OK;
}

int check_allocated(const kda_pool *p, const int32_t *ids, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        if (p->ref[ids[i]] < 1) return KDA_EREF;
    }
    return KDA_OK;
}

// Workspace: [SeqMeta][CkptMeta][pages][split items][wave offsets] (the uploaded metadata),
// then for the split path [operand images: 2 slots][wave state scratch][final windows].
struct WsLayout {
    int64_t o_ck = 0, o_pg = 0, o_items = 0, o_wso = 0, meta = 0;
    int64_t o_img = 0, o_state = 0, o_win = 0, total = 0;
};

WsLayout ws_layout(int64_t H, int64_t nseq, int64_t nck, int64_t P, const kda::SplitPlan *pl) {
    WsLayout L;
    L.o_ck = align_up(nseq * (int64_t)sizeof(SeqMeta), 256);
    L.o_pg = L.o_ck + align_up(nck * (int64_t)sizeof(CkptMeta), 256);
    L.o_items = L.o_pg + align_up((nseq + nck) * P * 4, 256);
    const int64_t nit = pl ? (int64_t)pl->items.size() : 0;
    L.o_wso = L.o_items + align_up(nit * (int64_t)sizeof(kda::SplitItem), 256);
    L.meta = L.o_wso + (pl ? (int64_t)pl->wave_seq_off.size() * 4 : 0);
    L.total = L.meta;
    if (pl) {
        L.o_img = align_up(L.meta, 1024);
        L.o_state = L.o_img + 2 * pl->slot_items * H * kda::kImageBytes;
        const int64_t state = pl->nwaves > 1 ? nseq * H * 128 * 128 * 4 : 0;
        L.o_win = L.o_state + state;
        L.total = L.o_win + nseq * H * 9 * 128 * 2;
    }
    return L;
}

// Metadata-only workspace of the fused kernels (also the layout the allocation-free path uses).
int64_t prefill_ws_bytes(int64_t nseq, int64_t nck, int64_t P) { return ws_layout(1, nseq, nck, P, nullptr).total; }

int copy_objects(kda_pool *p, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *src,
                 const int32_t *dst, void *pool_base, void *ws, int64_t ws_bytes, int32_t *status,
                 cudaStream_t stream) {
    const int32_t P = kda_object_pages(p, H, d, dtype);
    const int64_t list = (int64_t)n * P * 4;
    std::vector<int32_t> both((size_t)n * P * 2);
    std::memcpy(both.data(), src, (size_t)list);
    std::memcpy(both.data() + (size_t)n * P, dst, (size_t)list);
    int rc = kda::stage_upload(p, both.data(), (size_t)(2 * list), ws, stream);
    if (rc != KDA_OK) return rc;
    kda::CopyArgs a{};
    a.n = n;
    a.object_bytes = kda_object_bytes(H, d, dtype);
    a.pool = kda::pool_view(p, pool_base, H, d, dtype);
    a.src_pages = static_cast<const int32_t *>(ws);
    a.dst_pages = static_cast<const int32_t *>(ws) + (size_t)n * P;
    a.status = status;
    return kda::launch_copy_objects(a, stream) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

}  // namespace

namespace kda {

PoolView pool_view(const kda_pool *p, void *base, int32_t H, int32_t d, int32_t dtype) {
    PoolView v;
    v.base = static_cast<uint8_t *>(base);
    v.page_bytes = p->page_bytes;
    v.num_pages = p->num_pages;
    v.pages_per_object = kda_object_pages(p, H, d, dtype);
    v.rec_bytes = kda_record_bytes(d, dtype);
    v.page_shift = -1;
    for (int32_t sh = 0; sh < 63; ++sh)
        if (((int64_t)1 << sh) == p->page_bytes) v.page_shift = sh;
    // pages of 4 GiB or more: every in-object offset (below 4 GiB) is on page 0, which the
    // multiply gives with a zero reciprocal
    v.page_magic = p->page_bytes < ((int64_t)1 << 32)
                       ? (uint32_t)((((uint64_t)1 << 32) + (uint64_t)p->page_bytes - 1) / (uint64_t)p->page_bytes)
                       : 0u;
    return v;
}

}  // namespace kda

extern "C" {

int64_t kda_record_bytes(int32_t d, int32_t dtype) {
    if (!valid_shape(1, d, dtype)) return KDA_EINVAL;
    return align_up((int64_t)d * d * 4 + (int64_t)kda::kWin * 3 * d * elem_size(dtype), 256);
}

int64_t kda_object_bytes(int32_t H, int32_t d, int32_t dtype) {
    if (!valid_shape(H, d, dtype)) return KDA_EINVAL;
    return (int64_t)H * kda_record_bytes(d, dtype);
}

int32_t kda_object_pages(const kda_pool *p, int32_t H, int32_t d, int32_t dtype) {
    if (!p || !valid_shape(H, d, dtype)) return KDA_EINVAL;
    return (int32_t)((kda_object_bytes(H, d, dtype) + p->page_bytes - 1) / p->page_bytes);
}

int32_t kda_ckpt_positions(int64_t start, int64_t end, int32_t hash_block, int32_t stride,
                           int32_t include_last, int64_t *out, int32_t cap) {
    if (start < 0 || end < start || hash_block <= 0 || stride <= 0 || cap < 0 || (cap > 0 && !out))
        return KDA_EINVAL;
    const int64_t step = (int64_t)hash_block * stride;
    int64_t count = 0;
    int64_t last_emitted = -1;
    for (int64_t p = (start / step + 1) * step; p <= end; p += step) {
        if (count < cap) out[count] = p;
        ++count;
        last_emitted = p;
    }
    if (include_last) {
        const int64_t last = (end / hash_block) * hash_block;
        if (last > start && last != last_emitted) {
            if (count < cap) out[count] = last;   // last >= every stride multiple <= end
            ++count;
        }
    }
    if (count > INT32_MAX) return KDA_EINVAL;
    return (int32_t)count;
}

int kda_ckpt_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                  const int32_t *cu_seqlens, const int64_t *start_pos, int32_t hash_block,
                  int32_t stride, int32_t include_last, int32_t cap, int32_t *out_n,
                  int32_t *out_seq, int64_t *out_pos, int32_t *out_pages) {
    if (!pool || !valid_shape(H, d, dtype) || nseq < 0 || !cu_seqlens || !start_pos || !out_n ||
        hash_block <= 0 || hash_block % kda::kChunk != 0 || stride <= 0 || cap < 0)
        return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    std::vector<std::pair<int32_t, int64_t>> items;
    for (int32_t s = 0; s < nseq; ++s) {
        const int64_t len = (int64_t)cu_seqlens[s + 1] - cu_seqlens[s];
        if (len < 0 || start_pos[s] < 0) return KDA_EINVAL;
        const int32_t cnt = kda_ckpt_positions(start_pos[s], start_pos[s] + len, hash_block, stride,
                                               include_last, nullptr, 0);
        if (cnt < 0) return cnt;
        std::vector<int64_t> pos((size_t)cnt);
        kda_ckpt_positions(start_pos[s], start_pos[s] + len, hash_block, stride, include_last,
                           pos.data(), cnt);
        for (int64_t p : pos) items.emplace_back(s, p);
    }
    if ((int64_t)items.size() > cap) return KDA_EINVAL;
    if (!items.empty() && (!out_seq || !out_pos || !out_pages)) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    if ((int64_t)pool->free_n < (int64_t)items.size() * P) return KDA_ENOPAGES;
    for (size_t i = 0; i < items.size(); ++i) {
        out_seq[i] = items[i].first;
        out_pos[i] = items[i].second;
        kda::pool_alloc(pool, P, out_pages + i * (size_t)P);
    }
    *out_n = (int32_t)items.size();
    return KDA_OK;
}

int64_t kda_prefill_workspace_bytes(int32_t H, int32_t d, int32_t dtype, int32_t nseq, const int32_t *cu_seqlens,
                                    const int64_t *start_pos, int32_t n_ckpt, int32_t pages_per_object) {
    if (!valid_shape(H, d, dtype) || nseq < 0 || n_ckpt < 0 || pages_per_object <= 0) return KDA_EINVAL;
    if (!split_applies(d, dtype)) return prefill_ws_bytes(nseq, n_ckpt, pages_per_object);
    if (nseq > 0 && (!cu_seqlens || !start_pos)) return KDA_EINVAL;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || start_pos[s] < 0) return KDA_EINVAL;
    kda::SplitPlan pl;
    make_split_plan(H, nseq, cu_seqlens, start_pos, pl);
    return ws_layout(H, nseq, n_ckpt, pages_per_object, &pl).total;
}

int32_t kda_prefill_kernel_launches(int32_t H, int32_t d, int32_t dtype, int32_t nseq, const int32_t *cu_seqlens,
                                    const int64_t *start_pos) {
    if (!valid_shape(H, d, dtype) || nseq < 0) return KDA_EINVAL;
    if (!split_applies(d, dtype)) return 1;
    if (nseq > 0 && (!cu_seqlens || !start_pos)) return KDA_EINVAL;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || start_pos[s] < 0) return KDA_EINVAL;
    kda::SplitPlan pl;
    make_split_plan(H, nseq, cu_seqlens, start_pos, pl);
    // chunk preparation and chains per wave; every wave has at least one item
    return pl.nwaves == 0 ? 1 : 2 * pl.nwaves;
}

int32_t kda_prefill_waves(int32_t H, int32_t d, int32_t dtype, int32_t nseq, const int32_t *cu_seqlens,
                          const int64_t *start_pos, int32_t *wave_c0, int32_t cap) {
    if (!valid_shape(H, d, dtype) || nseq < 0 || cap < 0 || (cap > 0 && !wave_c0)) return KDA_EINVAL;
    if (nseq > 0 && (!cu_seqlens || !start_pos)) return KDA_EINVAL;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || start_pos[s] < 0) return KDA_EINVAL;
    if (!split_applies(d, dtype)) return 0;
    kda::SplitPlan pl;
    make_split_plan(H, nseq, cu_seqlens, start_pos, pl);
    for (int32_t i = 0; i < cap && i < (int32_t)pl.wave_c0.size(); ++i) wave_c0[i] = pl.wave_c0[i];
    return pl.nwaves;
}

int kda_prefill_varlen(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                       const int32_t *cu_seqlens, const int64_t *start_pos,
                       const uint8_t *has_init, const void *q, const void *k, const void *v,
                       const void *alpha, const void *beta, const float *conv_w, void *o,
                       void *pool_base, const int32_t *active_pages, int32_t n_ckpt,
                       const int32_t *ckpt_seq, const int64_t *ckpt_pos,
                       const int32_t *ckpt_pages, void *workspace, int64_t ws_bytes,
                       int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || nseq < 1 || !cu_seqlens || !start_pos || !has_init ||
        !conv_w || !pool_base || !active_pages || n_ckpt < 0 || !workspace || !status_dev)
        return KDA_EINVAL;
    if (n_ckpt > 0 && (!ckpt_seq || !ckpt_pos || !ckpt_pages)) return KDA_EINVAL;
    if (cu_seqlens[0] != 0) return KDA_EINVAL;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || start_pos[s] < 0 || has_init[s] > 1) return KDA_EINVAL;
    const int64_t T_tot = cu_seqlens[nseq];
    if ((int64_t)T_tot * H * d > ((int64_t)1 << 40)) return KDA_EINVAL;
    if (T_tot > 0 && (!q || !k || !v || !alpha || !beta || !o)) return KDA_EINVAL;
    if ((uintptr_t)workspace % 16 != 0) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    const bool split = split_applies(d, dtype);
    kda::SplitPlan plan;
    if (split) make_split_plan(H, nseq, cu_seqlens, start_pos, plan);
    const WsLayout L = ws_layout(H, nseq, n_ckpt, P, split ? &plan : nullptr);
    if (ws_bytes < L.total) return KDA_EINVAL;

    std::vector<SeqMeta> seqs((size_t)nseq);
    std::vector<CkptMeta> cks((size_t)n_ckpt);
    std::vector<int32_t> pages((size_t)(nseq + n_ckpt) * P);
    {
        std::lock_guard<std::mutex> g(pool->mu);
        const uint32_t gen = kda::pool_new_stamp(pool);
        int rc = check_private(pool, active_pages, (int64_t)nseq * P, gen);
        if (rc != KDA_OK) return rc;
        rc = check_private(pool, ckpt_pages, (int64_t)n_ckpt * P, gen);
        if (rc != KDA_OK) return rc;
    }
    std::memcpy(pages.data(), active_pages, (size_t)nseq * P * 4);
    if (n_ckpt) std::memcpy(pages.data() + (size_t)nseq * P, ckpt_pages, (size_t)n_ckpt * P * 4);
    int32_t ci = 0;
    for (int32_t s = 0; s < nseq; ++s) {
        SeqMeta &m = seqs[s];
        m.start_pos = start_pos[s];
        m.tok_begin = cu_seqlens[s];
        m.len = cu_seqlens[s + 1] - cu_seqlens[s];
        m.has_init = has_init[s];
        m.active_off = s * P;
        m.ckpt_begin = ci;
        const int64_t end = m.start_pos + m.len;
        int64_t prev = m.start_pos;
        while (ci < n_ckpt && ckpt_seq[ci] == s) {
            const int64_t p = ckpt_pos[ci];
            if (p <= prev || p > end || (p % kda::kChunk != 0 && p != end)) return KDA_EINVAL;
            cks[ci].pos = p;
            cks[ci].seq = s;
            cks[ci].pages_off = (nseq + ci) * P;
            prev = p;
            ++ci;
        }
        m.ckpt_count = ci - m.ckpt_begin;
    }
    if (ci != n_ckpt) return KDA_EINVAL;   // sequence ids not ascending or out of range
    if (split) {
        // each chunk-prep item learns here whether a checkpoint ends its chunk (its window is
        // written then), instead of searching the checkpoint table on the device
        for (kda::SplitItem &it : plan.items) {
            const SeqMeta &m = seqs[it.seq];
            const int64_t c_end = std::min<int64_t>(m.start_pos + m.len, (m.start_pos / kda::kChunk + it.lc + 1) * kda::kChunk);
            const auto b = cks.begin() + m.ckpt_begin, e = b + m.ckpt_count;   // positions ascend
            const auto f = std::lower_bound(b, e, c_end, [](const CkptMeta &c, int64_t p) { return c.pos < p; });
            it.ckpt = (f != e && f->pos == c_end) ? (int32_t)(f - cks.begin()) : -1;
        }
    }

    // One upload of the metadata part of the workspace layout.
    std::vector<uint8_t> blob((size_t)L.meta, 0);
    std::memcpy(blob.data(), seqs.data(), seqs.size() * sizeof(SeqMeta));
    if (n_ckpt) std::memcpy(blob.data() + L.o_ck, cks.data(), cks.size() * sizeof(CkptMeta));
    std::memcpy(blob.data() + L.o_pg, pages.data(), pages.size() * 4);
    if (split) {
        if (!plan.items.empty())
            std::memcpy(blob.data() + L.o_items, plan.items.data(), plan.items.size() * sizeof(kda::SplitItem));
        if (!plan.wave_seq_off.empty())
            std::memcpy(blob.data() + L.o_wso, plan.wave_seq_off.data(), plan.wave_seq_off.size() * 4);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = kda::stage_upload(pool, blob.data(), (size_t)L.meta, workspace, st);
    if (rc != KDA_OK) return rc;

    kda::PrefillArgs a{};
    a.H = H; a.d = d; a.dtype = dtype; a.nseq = nseq;
    a.T_tot = T_tot;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.conv_w = conv_w; a.o = o;
    a.pool = kda::pool_view(pool, pool_base, H, d, dtype);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.seqs = reinterpret_cast<const SeqMeta *>(ws);
    a.ckpts = reinterpret_cast<const CkptMeta *>(ws + L.o_ck);
    a.pages = reinterpret_cast<const int32_t *>(ws + L.o_pg);
    a.status = status_dev;
    if (!split) return kda::launch_prefill(a, st) == cudaSuccess ? KDA_OK : KDA_ECUDA;
    kda::SplitArgs sa;
    sa.p = a;
    sa.items = reinterpret_cast<const kda::SplitItem *>(ws + L.o_items);
    sa.wave_seq_off = reinterpret_cast<const int32_t *>(ws + L.o_wso);
    sa.images = ws + L.o_img;
    sa.slot_items = plan.slot_items;
    sa.state_scr = reinterpret_cast<float *>(ws + L.o_state);
    sa.win_scr = ws + L.o_win;
    sa.nwaves = plan.nwaves;
    return kda::launch_prefill_split(sa, plan, st) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

int kda_decode_step_pp(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, const void *q,
                       const void *k, const void *v, const void *alpha, const void *beta, const float *conv_w,
                       void *o, void *pool_base, const int32_t *src_pages, const int32_t *dst_pages,
                       int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || B < 0 || (int64_t)B * H > INT32_MAX || !status_dev)
        return KDA_EINVAL;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !alpha || !beta || !conv_w || !o || !pool_base || !src_pages || !dst_pages)
        return KDA_EINVAL;
    kda::DecodeArgs a{};
    a.H = H; a.d = d; a.dtype = dtype; a.B = B;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.conv_w = conv_w; a.o = o;
    a.pool = kda::pool_view(pool, pool_base, H, d, dtype);
    a.state_pages = src_pages;
    a.dst_pages = dst_pages;
    a.status = status_dev;
    return kda::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

int kda_decode_step(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, const void *q,
                    const void *k, const void *v, const void *alpha, const void *beta, const float *conv_w, void *o,
                    void *pool_base, const int32_t *state_pages, int32_t *status_dev, void *stream) {
    return kda_decode_step_pp(pool, H, d, dtype, B, q, k, v, alpha, beta, conv_w, o, pool_base, state_pages,
                              state_pages, status_dev, stream);
}

int kda_verify_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K,
                    int32_t *inter_pages_out) {
    if (!pool || !valid_shape(H, d, dtype) || B < 0 || K < 1 || K > 64 || (B > 0 && !inter_pages_out))
        return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    const int64_t need = (int64_t)B * K * P;
    if (need > INT32_MAX) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    if ((int64_t)pool->free_n < need) return KDA_ENOPAGES;
    return need ? kda::pool_alloc(pool, (int32_t)need, inter_pages_out) : KDA_OK;
}

int kda_verify_step(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K, const void *q,
                    const void *k, const void *v, const void *alpha, const void *beta, const float *conv_w, void *o,
                    void *pool_base, const int32_t *src_pages, const int32_t *inter_pages, int32_t *status_dev,
                    void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || B < 0 || K < 1 || K > 64 || !status_dev) return KDA_EINVAL;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !alpha || !beta || !conv_w || !o || !pool_base || !src_pages || !inter_pages)
        return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    {
        // one fused kernel where it applies: each source record read once, the state kept on
        // chip across the K draft tokens
        kda::VerifyArgs a{};
        a.H = H; a.d = d; a.dtype = dtype; a.B = B; a.K = K;
        a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.conv_w = conv_w; a.o = o;
        a.pool = kda::pool_view(pool, pool_base, H, d, dtype);
        a.src_pages = src_pages;
        a.inter_pages = inter_pages;
        a.status = status_dev;
        if (kda::verify_fused_supported(a))
            return kda::launch_verify_fused(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK : KDA_ECUDA;
    }
    // otherwise K stream-ordered ping-pong decode steps
    const int64_t e = elem_size(dtype), tok = (int64_t)B * H * d * e, btok = (int64_t)B * H * e;
    for (int32_t j = 0; j < K; ++j) {
        // draft token j of every request: state from the previous token's object (or the
        // source), written to this token's object
        const int32_t *src = j == 0 ? src_pages : inter_pages + (int64_t)(j - 1) * B * P;
        const int32_t *dst = inter_pages + (int64_t)j * B * P;
        auto at = [&](const void *base, int64_t stride) {
            return static_cast<const void *>(static_cast<const uint8_t *>(base) + j * stride);
        };
        const int rc = kda_decode_step_pp(pool, H, d, dtype, B, at(q, tok), at(k, tok), at(v, tok), at(alpha, tok),
                                          at(beta, btok), conv_w, static_cast<uint8_t *>(o) + j * tok, pool_base,
                                          src, dst, status_dev, stream);
        if (rc != KDA_OK) return rc;
    }
    return KDA_OK;
}

int kda_verify_accept(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K,
                      const int32_t *accepted, const int32_t *src_pages, const int32_t *inter_pages,
                      int32_t *active_out) {
    if (!pool || !valid_shape(H, d, dtype) || B < 0 || K < 1 || K > 64) return KDA_EINVAL;
    if (B == 0) return KDA_OK;
    if (!accepted || !src_pages || !inter_pages || !active_out) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    for (int32_t b = 0; b < B; ++b)
        if (accepted[b] < 0 || accepted[b] > K) return KDA_EINVAL;
    std::vector<int32_t> drop;
    drop.reserve((size_t)B * K * P);
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t j = -1; j < K; ++j) {   // j = -1: the source object
            const int32_t *obj = j < 0 ? src_pages + (int64_t)b * P : inter_pages + ((int64_t)j * B + b) * P;
            if (j + 1 == accepted[b]) std::memcpy(active_out + (int64_t)b * P, obj, (size_t)P * 4);
            else drop.insert(drop.end(), obj, obj + P);
        }
    }
    std::lock_guard<std::mutex> g(pool->mu);
    return kda::pool_decref(pool, (int32_t)drop.size(), drop.data());
}

int kda_decode_pingpong_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, const int64_t *pos,
                             int32_t interval, const int32_t *active_pages, int32_t *dst_pages_out,
                             int32_t *donated_out, int32_t *n_donated_out) {
    if (!pool || !valid_shape(H, d, dtype) || B < 0 || interval <= 0 || !n_donated_out) return KDA_EINVAL;
    *n_donated_out = 0;
    if (B == 0) return KDA_OK;
    if (!pos || !active_pages || !dst_pages_out || !donated_out) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    std::vector<int32_t> due;
    for (int32_t r = 0; r < B; ++r) {
        if (pos[r] < 0) return KDA_EINVAL;
        if (pos[r] > 0 && pos[r] % interval == 0) due.push_back(r);
    }
    std::lock_guard<std::mutex> g(pool->mu);
    const uint32_t gen = kda::pool_new_stamp(pool);
    int rc = check_private(pool, active_pages, (int64_t)B * P, gen);
    if (rc != KDA_OK) return rc;
    if ((int64_t)pool->free_n < (int64_t)due.size() * P) return KDA_ENOPAGES;
    std::memcpy(dst_pages_out, active_pages, (size_t)B * P * 4);
    for (size_t i = 0; i < due.size(); ++i) {
        kda::pool_alloc(pool, P, dst_pages_out + (size_t)due[i] * P);
        donated_out[i] = due[i];
    }
    *n_donated_out = (int32_t)due.size();
    return KDA_OK;
}

int64_t kda_copy_workspace_bytes(int32_t n, int32_t pages_per_object) {
    if (n < 0 || pages_per_object <= 0) return KDA_EINVAL;
    return align_up((int64_t)n * pages_per_object * 8, 256);
}

int kda_ckpt_write(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                   const int32_t *src_pages, int32_t *dst_pages_out, void *pool_base,
                   void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev)
        return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!src_pages || !dst_pages_out) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = check_allocated(pool, src_pages, (int64_t)n * P);
    if (rc != KDA_OK) return rc;
    rc = kda::pool_alloc(pool, n * P, dst_pages_out);
    if (rc != KDA_OK) return rc;
    rc = copy_objects(pool, H, d, dtype, n, src_pages, dst_pages_out, pool_base, workspace, ws_bytes,
                      status_dev, static_cast<cudaStream_t>(stream));
    if (rc != KDA_OK) kda::pool_decref(pool, n * P, dst_pages_out);
    return rc;
}

int kda_ckpt_restore(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                     const int32_t *ckpt_pages, const int32_t *active_pages, void *pool_base,
                     void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev)
        return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!ckpt_pages || !active_pages) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = check_allocated(pool, ckpt_pages, (int64_t)n * P);
    if (rc != KDA_OK) return rc;
    const uint32_t gen = kda::pool_new_stamp(pool);
    rc = check_private(pool, active_pages, (int64_t)n * P, gen);
    if (rc != KDA_OK) return rc;
    for (int64_t i = 0; i < (int64_t)n * P; ++i)
        if (pool->stamp[ckpt_pages[i]] == gen) return KDA_EREF;   // never copy onto the source
    rc = kda::pool_incref(pool, n * P, ckpt_pages);
    if (rc != KDA_OK) return rc;
    rc = copy_objects(pool, H, d, dtype, n, ckpt_pages, active_pages, pool_base, workspace, ws_bytes,
                      status_dev, static_cast<cudaStream_t>(stream));
    if (rc != KDA_OK) kda::pool_decref(pool, n * P, ckpt_pages);
    return rc;
}

int kda_ckpt_release(kda_pool *pool, int32_t n, int32_t pages_per_object, const int32_t *ckpt_pages) {
    if (!pool || n < 0 || pages_per_object <= 0) return KDA_EINVAL;
    return kda_page_decref(pool, n * pages_per_object, ckpt_pages);
}

int64_t kda_record_bytes_q8(int32_t d, int32_t dtype) {
    if (!valid_shape(1, d, dtype)) return KDA_EINVAL;
    return align_up((int64_t)4 * d + (int64_t)d * d + (int64_t)kda::kWin * 3 * d * elem_size(dtype), 256);
}

int64_t kda_object_bytes_q8(int32_t H, int32_t d, int32_t dtype) {
    if (!valid_shape(H, d, dtype)) return KDA_EINVAL;
    return (int64_t)H * kda_record_bytes_q8(d, dtype);
}

int32_t kda_object_pages_q8(const kda_pool *p, int32_t H, int32_t d, int32_t dtype) {
    if (!p || !valid_shape(H, d, dtype)) return KDA_EINVAL;
    return (int32_t)((kda_object_bytes_q8(H, d, dtype) + p->page_bytes - 1) / p->page_bytes);
}

}  // extern "C"

namespace {

// Upload [full lists][q8 lists] and run one conversion (quantise or dequantise).
int convert_q8(kda_pool *p, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *full,
               const int32_t *q8, void *pool_base, void *ws, int32_t *status, cudaStream_t stream, bool quantize) {
    const int32_t P = kda_object_pages(p, H, d, dtype), Pq = kda_object_pages_q8(p, H, d, dtype);
    std::vector<int32_t> both((size_t)n * (P + Pq));
    std::memcpy(both.data(), full, (size_t)n * P * 4);
    std::memcpy(both.data() + (size_t)n * P, q8, (size_t)n * Pq * 4);
    int rc = kda::stage_upload(p, both.data(), both.size() * 4, ws, stream);
    if (rc != KDA_OK) return rc;
    kda::Q8Args a{};
    a.n = n;
    a.H = H;
    a.d = d;
    a.dtype = dtype;
    a.full = kda::pool_view(p, pool_base, H, d, dtype);
    a.q8 = a.full;
    a.q8.pages_per_object = Pq;
    a.q8.rec_bytes = kda_record_bytes_q8(d, dtype);
    a.full_pages = static_cast<const int32_t *>(ws);
    a.q8_pages = static_cast<const int32_t *>(ws) + (size_t)n * P;
    a.status = status;
    const cudaError_t e = quantize ? kda::launch_ckpt_quantize(a, stream) : kda::launch_ckpt_dequantize(a, stream);
    return e == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

bool q8_sizes_ok(const kda_pool *p, int32_t H, int32_t d, int32_t dtype) {
    return p->page_bytes < ((int64_t)1 << 32) && kda_object_bytes(H, d, dtype) < ((int64_t)1 << 32);
}

}  // namespace

extern "C" {

int kda_ckpt_write_q8(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *src_pages,
                      int32_t *dst_pages_out, void *pool_base, void *workspace, int64_t ws_bytes,
                      int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev) return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!src_pages || !dst_pages_out || !q8_sizes_ok(pool, H, d, dtype)) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype), Pq = kda_object_pages_q8(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = check_allocated(pool, src_pages, (int64_t)n * P);
    if (rc != KDA_OK) return rc;
    rc = kda::pool_alloc(pool, n * Pq, dst_pages_out);
    if (rc != KDA_OK) return rc;
    rc = convert_q8(pool, H, d, dtype, n, src_pages, dst_pages_out, pool_base, workspace, status_dev,
                    static_cast<cudaStream_t>(stream), true);
    if (rc != KDA_OK) kda::pool_decref(pool, n * Pq, dst_pages_out);
    return rc;
}

int kda_ckpt_restore_q8(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *ckpt_pages,
                        const int32_t *active_pages, void *pool_base, void *workspace, int64_t ws_bytes,
                        int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev) return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!ckpt_pages || !active_pages || !q8_sizes_ok(pool, H, d, dtype)) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype), Pq = kda_object_pages_q8(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = check_allocated(pool, ckpt_pages, (int64_t)n * Pq);
    if (rc != KDA_OK) return rc;
    const uint32_t gen = kda::pool_new_stamp(pool);
    rc = check_private(pool, active_pages, (int64_t)n * P, gen);
    if (rc != KDA_OK) return rc;
    for (int64_t i = 0; i < (int64_t)n * Pq; ++i)
        if (pool->stamp[ckpt_pages[i]] == gen) return KDA_EREF;   // never convert onto the source
    rc = kda::pool_incref(pool, n * Pq, ckpt_pages);
    if (rc != KDA_OK) return rc;
    rc = convert_q8(pool, H, d, dtype, n, active_pages, ckpt_pages, pool_base, workspace, status_dev,
                    static_cast<cudaStream_t>(stream), false);
    if (rc != KDA_OK) kda::pool_decref(pool, n * Pq, ckpt_pages);
    return rc;
}

}  // extern "C"

namespace {

// Device address of a pinned, mapped host buffer (nullptr when it is not device-accessible).
void *host_device_ptr(void *host) {
    void *dev = nullptr;
    if (cudaHostGetDevicePointer(&dev, host, 0) != cudaSuccess) {
        cudaGetLastError();   // the failed query leaves a (non-sticky) error: clear it
        return nullptr;
    }
    return dev;
}

int host_copy(kda_pool *p, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *pages, void *host,
              void *pool_base, void *ws, int32_t *status, cudaStream_t stream, bool to_host) {
    const int32_t P = kda_object_pages(p, H, d, dtype);
    int rc = kda::stage_upload(p, pages, (size_t)n * P * 4, ws, stream);
    if (rc != KDA_OK) return rc;
    kda::HostCopyArgs a{};
    a.n = n;
    a.object_bytes = kda_object_bytes(H, d, dtype);
    a.pool = kda::pool_view(p, pool_base, H, d, dtype);
    a.pages = static_cast<const int32_t *>(ws);
    a.host = static_cast<uint8_t *>(host);
    a.to_host = to_host ? 1 : 0;
    a.status = status;
    return kda::launch_host_copy(a, stream) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

}  // namespace

extern "C" {

int kda_ckpt_offload(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n, const int32_t *pages,
                     void *host_dst, int64_t host_bytes, void *pool_base, void *workspace, int64_t ws_bytes,
                     int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev) return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!pages || !host_dst || host_bytes < (int64_t)n * kda_object_bytes(H, d, dtype)) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0 || (uintptr_t)host_dst % 16 != 0)
        return KDA_EINVAL;
    void *dev = host_device_ptr(host_dst);
    if (!dev) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = check_allocated(pool, pages, (int64_t)n * P);
    if (rc != KDA_OK) return rc;
    return host_copy(pool, H, d, dtype, n, pages, dev, pool_base, workspace, status_dev,
                     static_cast<cudaStream_t>(stream), true);
}

int kda_ckpt_prefetch(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n, const void *host_src,
                      int64_t host_bytes, int32_t *pages_out, void *pool_base, void *workspace, int64_t ws_bytes,
                      int32_t *status_dev, void *stream) {
    if (!pool || !valid_shape(H, d, dtype) || n < 0 || !pool_base || !workspace || !status_dev) return KDA_EINVAL;
    if (n == 0) return KDA_OK;
    if (!pages_out || !host_src || host_bytes < (int64_t)n * kda_object_bytes(H, d, dtype)) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    if (ws_bytes < kda_copy_workspace_bytes(n, P) || (uintptr_t)workspace % 16 != 0 || (uintptr_t)host_src % 16 != 0)
        return KDA_EINVAL;
    void *dev = host_device_ptr(const_cast<void *>(host_src));
    if (!dev) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(pool->mu);
    int rc = kda::pool_alloc(pool, n * P, pages_out);
    if (rc != KDA_OK) return rc;
    rc = host_copy(pool, H, d, dtype, n, pages_out, dev, pool_base, workspace, status_dev,
                   static_cast<cudaStream_t>(stream), false);
    if (rc != KDA_OK) kda::pool_decref(pool, n * P, pages_out);
    return rc;
}

int kda_sync_status(int32_t *status_dev, void *stream, int32_t *bits_out) {
    if (!status_dev) return KDA_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, status_dev, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KDA_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ECUDA;
    if (bits_out) *bits_out = h;
    if (h != 0) {
        if (cudaMemsetAsync(status_dev, 0, 4, st) != cudaSuccess) return KDA_ECUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ECUDA;
        return KDA_EDEVICE;
    }
    return KDA_OK;
}

const char *kda_status_string(int code) {
    switch (code) {
        case KDA_OK: return "ok";
        case KDA_EINVAL: return "invalid argument";
        case KDA_ENOPAGES: return "page pool exhausted";
        case KDA_EREF: return "reference-count misuse";
        case KDA_ECUDA: return "CUDA error";
        case KDA_EDEVICE: return "device-side check failed";
        default: return "unknown status";
    }
}

}  // extern "C"
