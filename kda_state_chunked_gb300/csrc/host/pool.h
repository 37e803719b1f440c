// Host-side page pool of libkda.so: one page byte size, lowest-free-first allocation,
// reference counts, and pinned staging buffers that carry call metadata to the device.
#pragma once

#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "../kda_internal.h"

struct kda_pool {
    int64_t page_bytes = 0;
    int32_t num_pages = 0;
    std::vector<int32_t> ref;        // reference count per page (0 = free)
    std::vector<uint64_t> free_bits; // bit i set <=> page i free
    int32_t free_n = 0;
    int32_t low_word = 0;            // no free page below word low_word
    std::vector<uint32_t> stamp;     // per-page marks for duplicate checks within one call
    uint32_t stamp_gen = 0;

    // Pinned host staging slots, reused round-robin; each slot's event marks the end of the
    // last host-to-device copy that read it.
    struct Slot {
        void *host = nullptr;
        size_t cap = 0;
        cudaEvent_t done = nullptr;
        bool pending = false;
    };
    static constexpr int kSlots = 4;
    Slot slots[kSlots];
    int next_slot = 0;
    std::mutex mu;
};

namespace kda {

void pool_mark_free(kda_pool *p, int32_t id);
void pool_mark_used(kda_pool *p, int32_t id);
// Start a new duplicate-check generation; returns the mark value for this call.
uint32_t pool_new_stamp(kda_pool *p);

// Allocator primitives (caller holds pool->mu).  All return a kda_status.
int pool_alloc(kda_pool *p, int32_t n, int32_t *out);
int pool_decref(kda_pool *p, int32_t n, const int32_t *ids);
int pool_incref(kda_pool *p, int32_t n, const int32_t *ids);

// Geometry of `p` for objects of H heads (d, dtype), with the page translation constants
// (shift for power-of-two page sizes, reciprocal otherwise) that every kernel uses.
PoolView pool_view(const kda_pool *p, void *base, int32_t H, int32_t d, int32_t dtype);

// Copy `bytes` of host data to device memory `dst` on `stream` through a pinned slot.
// The host data may be reused as soon as this returns.
int stage_upload(kda_pool *p, const void *src, size_t bytes, void *dst, cudaStream_t stream);

}  // namespace kda
