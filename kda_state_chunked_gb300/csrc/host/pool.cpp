// Page pool: the single allocator, reference-count and free-list implementation shared by
// every state object ("Cache de préfixe hybride KDA–MLA", §La mise en page unifiée: both
// page kinds share one implementation of allocation, reference counting and eviction).
#include "pool.h"

#include <cstring>
#include <unordered_map>

#include "kda.h"
#include "../kda_internal.h"

namespace kda {

int pool_alloc(kda_pool *p, int32_t n, int32_t *out) {
    if (n < 0 || (n > 0 && !out)) return KDA_EINVAL;
    if ((int64_t)p->free_ids.size() < n) return KDA_ENOPAGES;
    for (int32_t i = 0; i < n; ++i) {
        auto it = p->free_ids.begin();
        out[i] = *it;
        p->ref[*it] = 1;
        p->free_ids.erase(it);
    }
    return KDA_OK;
}

int pool_incref(kda_pool *p, int32_t n, const int32_t *ids) {
    if (n < 0 || (n > 0 && !ids)) return KDA_EINVAL;
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        if (p->ref[ids[i]] <= 0) return KDA_EREF;
    }
    for (int32_t i = 0; i < n; ++i) p->ref[ids[i]] += 1;
    return KDA_OK;
}

int pool_decref(kda_pool *p, int32_t n, const int32_t *ids) {
    if (n < 0 || (n > 0 && !ids)) return KDA_EINVAL;
    std::unordered_map<int32_t, int32_t> need;
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        need[ids[i]] += 1;
    }
    for (const auto &kv : need)
        if (p->ref[kv.first] < kv.second) return KDA_EREF;
    for (int32_t i = 0; i < n; ++i) {
        if (--p->ref[ids[i]] == 0) p->free_ids.insert(ids[i]);
    }
    return KDA_OK;
}

int stage_upload(kda_pool *p, const void *src, size_t bytes, void *dst, cudaStream_t stream) {
    if (bytes == 0) return KDA_OK;
    kda_pool::Slot &s = p->slots[p->next_slot];
    p->next_slot = (p->next_slot + 1) % kda_pool::kSlots;
    if (s.pending) {
        if (cudaEventSynchronize(s.done) != cudaSuccess) return KDA_ECUDA;
        s.pending = false;
    }
    if (!s.done && cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess)
        return KDA_ECUDA;
    if (s.cap < bytes) {
        if (s.host) cudaFreeHost(s.host);
        s.host = nullptr;
        s.cap = 0;
        size_t cap = bytes < 65536 ? 65536 : bytes * 2;
        if (cudaHostAlloc(&s.host, cap, cudaHostAllocPortable) != cudaSuccess) return KDA_ECUDA;
        s.cap = cap;
    }
    std::memcpy(s.host, src, bytes);
    if (cudaMemcpyAsync(dst, s.host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return KDA_ECUDA;
    if (cudaEventRecord(s.done, stream) != cudaSuccess) return KDA_ECUDA;
    s.pending = true;
    return KDA_OK;
}

}  // namespace kda

extern "C" {

int kda_pool_create(int64_t page_bytes, int32_t num_pages, kda_pool **out) {
    if (!out || page_bytes <= 0 || page_bytes % 256 != 0 || num_pages <= 0) return KDA_EINVAL;
    kda_pool *p = new (std::nothrow) kda_pool();
    if (!p) return KDA_ENOPAGES;
    p->page_bytes = page_bytes;
    p->num_pages = num_pages;
    p->ref.assign((size_t)num_pages, 0);
    for (int32_t i = 0; i < num_pages; ++i) p->free_ids.insert(p->free_ids.end(), i);
    *out = p;
    return KDA_OK;
}

int kda_pool_destroy(kda_pool *p) {
    if (!p) return KDA_EINVAL;
    for (auto &s : p->slots) {
        if (s.pending) cudaEventSynchronize(s.done);
        if (s.done) cudaEventDestroy(s.done);
        if (s.host) cudaFreeHost(s.host);
    }
    delete p;
    return KDA_OK;
}

int64_t kda_pool_page_bytes(const kda_pool *p) { return p ? p->page_bytes : KDA_EINVAL; }
int32_t kda_pool_num_pages(const kda_pool *p) { return p ? p->num_pages : KDA_EINVAL; }

int32_t kda_pool_free_count(const kda_pool *p) {
    if (!p) return KDA_EINVAL;
    return (int32_t)p->free_ids.size();
}

int kda_page_alloc(kda_pool *p, int32_t n, int32_t *out_ids) {
    if (!p) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    return kda::pool_alloc(p, n, out_ids);
}

int kda_page_claim(kda_pool *p, int32_t n, const int32_t *ids) {
    if (!p || n < 0 || (n > 0 && !ids)) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    std::set<int32_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        if (p->ref[ids[i]] != 0 || !seen.insert(ids[i]).second) return KDA_EREF;
    }
    for (int32_t i = 0; i < n; ++i) {
        p->ref[ids[i]] = 1;
        p->free_ids.erase(ids[i]);
    }
    return KDA_OK;
}

int kda_page_incref(kda_pool *p, int32_t n, const int32_t *ids) {
    if (!p) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    return kda::pool_incref(p, n, ids);
}

int kda_page_decref(kda_pool *p, int32_t n, const int32_t *ids) {
    if (!p) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    return kda::pool_decref(p, n, ids);
}

int32_t kda_page_refcount(const kda_pool *p, int32_t id) {
    if (!p || id < 0 || id >= p->num_pages) return KDA_EINVAL;
    return p->ref[id];
}

}  // extern "C"
