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
    // a shift for the usual power-of-two page sizes; a 64-bit division costs far more
    const uint64_t pi = pv.page_shift >= 0 ? off >> pv.page_shift : off / pb;
    const int32_t id = pages[pi];
    if ((uint32_t)id >= (uint32_t)pv.num_pages) {
        flag_status(status, KDA_DEV_BAD_PAGE);
        return nullptr;
    }
    return pv.base + (uint64_t)id * pb + (off - pi * pb);
}

// True when every page id of an object's list is inside the pool.
__device__ __forceinline__ bool pages_ok(const PoolView &pv, const int32_t *pages) {
    for (int i = 0; i < pv.pages_per_object; ++i)
        if ((uint32_t)pages[i] >= (uint32_t)pv.num_pages) return false;
    return true;
}

}  // namespace kda
