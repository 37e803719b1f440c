// kda_prefill_varlen_noalloc: the chunked varlen prefill for callers that cannot allocate
// device memory when they call it.
//
// kda_prefill_varlen needs a caller-provided device workspace for its per-call metadata
// (sequence table, checkpoint table, page lists).  Some callers cannot produce one at call
// time: a serving runtime that reserves all of HBM for its own pool at start-up (so a
// cudaMalloc there fails or fragments that pool), or a code path with a strict latency
// budget where cudaMalloc / cudaFree and the device synchronisation they can cause are
// not allowed.  This entry point keeps that metadata in a fixed array in the library's
// own device memory instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds
// KDA_NOALLOC_SCRATCH_BYTES of it until the process exits.  Its host-side name is only a
// handle, so the device address is looked up once per device (with that device current)
// by the first call on that device, and cached.
#include <cstring>
#include <mutex>

#include "kda.h"
#include "pool.h"
#include "../kda_internal.h"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Device-side scratch shared by every call on a device.
static __device__ __align__(256) uint8_t g_prefill_scratch[kScratchBytes];

// Host-side assembly buffer (static storage: no heap allocation per call).
alignas(256) static uint8_t g_host_meta[kScratchBytes];

std::mutex g_mu;                       // guards g_host_meta and g_dev_ptr
void *g_dev_ptr[kMaxDevices] = {};     // device address of g_prefill_scratch per device

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int kda_prefill_varlen_noalloc(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                                          const int32_t *cu_seqlens, const int64_t *start_pos,
                                          const uint8_t *has_init, const void *q, const void *k, const void *v,
                                          const void *alpha, const void *beta, const float *conv_w, void *o,
                                          void *pool_base, const int32_t *active_pages, int32_t n_ckpt,
                                          const int32_t *ckpt_seq, const int64_t *ckpt_pos,
                                          const int32_t *ckpt_pages, int32_t *status_dev, void *stream) {
    using kda::CkptMeta;
    using kda::SeqMeta;
    // Argument rules are those of kda_prefill_varlen.
    if (!pool || H <= 0 || H > 4096 || (d != 64 && d != 128) || (dtype != KDA_F32 && dtype != KDA_BF16) ||
        nseq < 1 || !cu_seqlens || !start_pos || !has_init || !conv_w || !pool_base || !active_pages ||
        n_ckpt < 0 || !status_dev)
        return KDA_EINVAL;
    if (n_ckpt > 0 && (!ckpt_seq || !ckpt_pos || !ckpt_pages)) return KDA_EINVAL;
    if (cu_seqlens[0] != 0) return KDA_EINVAL;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s] || start_pos[s] < 0 || has_init[s] > 1) return KDA_EINVAL;
    const int64_t T_tot = cu_seqlens[nseq];
    if (T_tot * H * d > ((int64_t)1 << 40)) return KDA_EINVAL;
    if (T_tot > 0 && (!q || !k || !v || !alpha || !beta || !o)) return KDA_EINVAL;
    const int32_t P = kda_object_pages(pool, H, d, dtype);
    if (P <= 0) return KDA_EINVAL;

    // Metadata layout in the scratch: [SeqMeta x nseq][CkptMeta x n_ckpt][int32 pages].
    const size_t o_ck = align256((size_t)nseq * sizeof(SeqMeta));
    const size_t o_pg = o_ck + align256((size_t)n_ckpt * sizeof(CkptMeta));
    const size_t total = o_pg + (size_t)(nseq + n_ckpt) * (size_t)P * 4;
    if (total > kScratchBytes) return KDA_EINVAL;   // more than the fixed scratch holds

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_EINVAL;

    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return KDA_ECUDA;
        g_dev_ptr[dev] = p;
    }
    {
        // Pages written by the call must be allocated, private (refcount 1) and distinct.
        std::lock_guard<std::mutex> g(pool->mu);
        const uint32_t gen = kda::pool_new_stamp(pool);
        const int32_t *lists[2] = {active_pages, ckpt_pages};
        const int64_t counts[2] = {(int64_t)nseq * P, (int64_t)n_ckpt * P};
        for (int l = 0; l < 2; ++l)
            for (int64_t i = 0; i < counts[l]; ++i) {
                const int32_t id = lists[l][i];
                if (id < 0 || id >= pool->num_pages) return KDA_EINVAL;
                if (pool->ref[id] != 1 || pool->stamp[id] == gen) return KDA_EREF;
                pool->stamp[id] = gen;
            }
    }
    std::memset(g_host_meta, 0, total);
    SeqMeta *seqs = reinterpret_cast<SeqMeta *>(g_host_meta);
    CkptMeta *cks = reinterpret_cast<CkptMeta *>(g_host_meta + o_ck);
    int32_t *pages = reinterpret_cast<int32_t *>(g_host_meta + o_pg);
    std::memcpy(pages, active_pages, (size_t)nseq * P * 4);
    if (n_ckpt) std::memcpy(pages + (size_t)nseq * P, ckpt_pages, (size_t)n_ckpt * P * 4);
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
    if (ci != n_ckpt) return KDA_EINVAL;

    // Pageable host source: the runtime copies it out before returning, so the static host
    // buffer is free for the next call once this returns.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(g_dev_ptr[dev], g_host_meta, total, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KDA_ECUDA;

    kda::PrefillArgs a{};
    a.H = H; a.d = d; a.dtype = dtype; a.nseq = nseq;
    a.T_tot = T_tot;
    a.q = q; a.k = k; a.v = v; a.alpha = alpha; a.beta = beta; a.conv_w = conv_w; a.o = o;
    // the same pool geometry (page translation constants included) as every other call
    a.pool = kda::pool_view(pool, pool_base, H, d, dtype);
    uint8_t *ws = static_cast<uint8_t *>(g_dev_ptr[dev]);
    a.seqs = reinterpret_cast<const SeqMeta *>(ws);
    a.ckpts = reinterpret_cast<const CkptMeta *>(ws + o_ck);
    a.pages = reinterpret_cast<const int32_t *>(ws + o_pg);
    a.status = status_dev;
    return kda::launch_prefill(a, st) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}
