// Page pool: the single allocator, reference-count and free-list implementation shared by
// every state object ("Cache de préfixe hybride KDA–MLA", §La mise en page unifiée: both
// page kinds share one implementation of allocation, reference counting and eviction).
#include "pool.h"

#include <algorithm>
#include <cstring>
#include <unordered_map>

#include "kda.h"
#include "../kda_internal.h"

namespace kda {

void pool_mark_free(kda_pool *p, int32_t id) {
    p->free_bits[(size_t)id >> 6] |= (uint64_t)1 << (id & 63);
    ++p->free_n;
    if ((id >> 6) < p->low_word) p->low_word = id >> 6;
}

void pool_mark_used(kda_pool *p, int32_t id) {
    p->free_bits[(size_t)id >> 6] &= ~((uint64_t)1 << (id & 63));
    --p->free_n;
}

uint32_t pool_new_stamp(kda_pool *p) {
    if (++p->stamp_gen == 0) {   // wrapped: clear all marks
        std::fill(p->stamp.begin(), p->stamp.end(), 0u);
        p->stamp_gen = 1;
    }
    return p->stamp_gen;
}

// Lowest free ids first: scan the free bitmap upward from the lowest word with a free bit.
int pool_alloc(kda_pool *p, int32_t n, int32_t *out) {
    if (n < 0 || (n > 0 && !out)) return KDA_EINVAL;
    if (p->free_n < n) return KDA_ENOPAGES;
    int32_t got = 0;
    size_t w = (size_t)p->low_word;
    while (got < n) {
        uint64_t bits = p->free_bits[w];
        while (bits && got < n) {
            const int b = __builtin_ctzll(bits);
            bits &= bits - 1;
            const int32_t id = (int32_t)(w * 64 + b);
            out[got++] = id;
            p->ref[id] = 1;
            p->free_bits[w] &= ~((uint64_t)1 << b);
        }
        if (got < n) ++w;
    }
    p->free_n -= n;
    while ((size_t)p->low_word < p->free_bits.size() && p->free_bits[p->low_word] == 0) ++p->low_word;
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
    // Count repeated ids against the refcount: stamp each id, and for ids seen more than once
    // in this call fall back to an exact count.
    const uint32_t g = pool_new_stamp(p);
    bool repeats = false;
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        if (p->ref[ids[i]] < 1) return KDA_EREF;
        if (p->stamp[ids[i]] == g) repeats = true;
        p->stamp[ids[i]] = g;
    }
    if (repeats) {
        std::unordered_map<int32_t, int32_t> need;
        for (int32_t i = 0; i < n; ++i) need[ids[i]] += 1;
        for (const auto &kv : need)
            if (p->ref[kv.first] < kv.second) return KDA_EREF;
    }
    for (int32_t i = 0; i < n; ++i) {
        if (--p->ref[ids[i]] == 0) pool_mark_free(p, ids[i]);
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
        // Grow every slot at once so that steady-state calls never allocate pinned memory.
        const size_t cap = bytes < ((size_t)1 << 20) ? ((size_t)1 << 20) : bytes * 2;
        for (auto &o : p->slots) {
            if (o.cap >= cap) continue;
            if (o.pending) {
                if (cudaEventSynchronize(o.done) != cudaSuccess) return KDA_ECUDA;
                o.pending = false;
            }
            if (o.host) cudaFreeHost(o.host);
            o.host = nullptr;
            o.cap = 0;
            if (cudaHostAlloc(&o.host, cap, cudaHostAllocPortable) != cudaSuccess) return KDA_ECUDA;
            o.cap = cap;
        }
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
    p->stamp.assign((size_t)num_pages, 0u);
    p->free_bits.assign(((size_t)num_pages + 63) / 64, ~(uint64_t)0);
    if (num_pages % 64) p->free_bits.back() = ((uint64_t)1 << (num_pages % 64)) - 1;
    p->free_n = num_pages;
    p->low_word = 0;
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
    return p->free_n;
}

int kda_page_alloc(kda_pool *p, int32_t n, int32_t *out_ids) {
    if (!p) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    return kda::pool_alloc(p, n, out_ids);
}

int kda_page_claim(kda_pool *p, int32_t n, const int32_t *ids) {
    if (!p || n < 0 || (n > 0 && !ids)) return KDA_EINVAL;
    std::lock_guard<std::mutex> g(p->mu);
    const uint32_t gen = kda::pool_new_stamp(p);
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= p->num_pages) return KDA_EINVAL;
        if (p->ref[ids[i]] != 0 || p->stamp[ids[i]] == gen) return KDA_EREF;
        p->stamp[ids[i]] = gen;
    }
    for (int32_t i = 0; i < n; ++i) {
        p->ref[ids[i]] = 1;
        kda::pool_mark_used(p, ids[i]);
    }
    while ((size_t)p->low_word < p->free_bits.size() && p->free_bits[p->low_word] == 0) ++p->low_word;
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
