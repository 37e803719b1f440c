// Host plan of the split bf16 prefill: which shapes take it and how a batch's chunks are cut
// into waves (one wave = chunk preparation of its (chunk, head) items, then the chains).
#pragma once

#include <cstdint>

#include "../kda_internal.h"

namespace kda {

// The split tensor-core prefill serves bf16 with d = 128; other shapes use one launch of the
// fused (fp32: CUDA-core) kernel and need metadata only.
bool split_applies(int32_t d, int32_t dtype);

// Chunks (aligned to absolute positions, 64 tokens) of a sequence of `len` tokens from `start`.
int32_t chunks_of(int64_t start, int64_t len);

// Waves of local chunks [wave_c0[w], wave_c0[w + 1]) of every chain, chosen by a cost model
// of the wave steps among splits that keep one slot of operand images (all chains' items of a
// wave) under 512 MiB.
void make_split_plan(int32_t H, int32_t nseq, const int32_t *cu, const int64_t *start, SplitPlan &pl);

}  // namespace kda
