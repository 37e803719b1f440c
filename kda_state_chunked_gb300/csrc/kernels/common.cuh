// Device helpers shared by the KDA kernels: element loads/stores in the token dtype and
// logical-offset -> page translation for state records in the paged pool.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

#include "../kda_internal.h"

namespace kda {

__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ void flag_status(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// Address of logical byte `off` of an object whose page list is `pages`.  Returns nullptr
// (and flags KDA_DEV_BAD_PAGE) when the page id lies outside the pool.  Callers keep every
// access of one call inside a 16-byte unit that never straddles pages (records and pages
// are multiples of 256 bytes).
__device__ __forceinline__ uint8_t *obj_addr(const PoolView &pv, const int32_t *pages,
                                             uint64_t off, int32_t *status) {
    const uint64_t pb = (uint64_t)pv.page_bytes;
    // Page index: a shift for power-of-two page sizes; otherwise off / pb without a division
    // (an object is below 4 GiB, so off fits 32 bits): q = high half of off * ceil(2^32 / pb)
    // is off / pb or one more, and one multiply-compare corrects it.
    uint64_t pi;
    if (pv.page_shift >= 0) {
        pi = off >> pv.page_shift;
    } else {
        const uint32_t o = (uint32_t)off;
        uint32_t q = __umulhi(o, pv.page_magic);
        if ((uint64_t)q * pb > o) --q;
        pi = q;
    }
    const int32_t id = pages[pi];
    if ((uint32_t)id >= (uint32_t)pv.num_pages) {
        flag_status(status, KDA_DEV_BAD_PAGE);
        return nullptr;
    }
    return pv.base + (uint64_t)id * pb + (off - pi * pb);
}

// Base address of a run of accesses at off0 .. off0 + span of one object when the run is
// contiguous in the pool (one page, or physically adjacent pages), so that every access in it
// is base + (off - off0); nullptr otherwise (the caller then translates each access).
__device__ __forceinline__ uint8_t *run_addr(const PoolView &pv, const int32_t *pages, uint64_t off0,
                                             uint64_t span, int32_t *status) {
    uint8_t *a = obj_addr(pv, pages, off0, status), *b = obj_addr(pv, pages, off0 + span, status);
    return (a && b && b - a == (int64_t)span) ? a : nullptr;
}

// True when every page id of an object's list is inside the pool.
__device__ __forceinline__ bool pages_ok(const PoolView &pv, const int32_t *pages) {
    for (int i = 0; i < pv.pages_per_object; ++i)
        if ((uint32_t)pages[i] >= (uint32_t)pv.num_pages) return false;
    return true;
}

}  // namespace kda
