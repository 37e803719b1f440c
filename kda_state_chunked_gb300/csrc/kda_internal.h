// Internal declarations shared by the host library and the CUDA kernels of libkda.so.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;   // tokens per chunk; chunks are aligned to absolute positions
constexpr int kConvW = 4;    // short causal conv width (taps on t-3 .. t)
constexpr int kWin = kConvW - 1;
// Smallest product of alpha over one chunk, per key channel, that the chunked prefill kernels
// accept: they scale rows by gamma_r / gamma_C (up to 1 / gamma_C) and by its inverse, which
// must stay far inside the fp32 / bf16 exponent range.  Below it a kernel sets KDA_DEV_RANGE.
constexpr float kMinChunkDecay = 0x1p-100f;

// Per-sequence metadata of one prefill call (device copy in the workspace).
struct SeqMeta {
    int64_t start_pos;   // absolute position of the first token
    int32_t tok_begin;   // row of the first token in the packed [T_tot][H][d] arrays
    int32_t len;         // tokens in this call
    int32_t has_init;    // 1: read (S, window) from the active object first
    int32_t ckpt_begin;  // first entry of this sequence in the checkpoint table
    int32_t ckpt_count;  // number of entries
    int32_t active_off;  // offset of the active object's page list in the page array
};
static_assert(sizeof(SeqMeta) == 32, "SeqMeta layout");

// One checkpoint to stream (device copy in the workspace).
struct CkptMeta {
    int64_t pos;         // absolute position p: state after tokens [0, p)
    int32_t pages_off;   // offset of its page list in the page array
    int32_t seq;         // owning sequence
};
static_assert(sizeof(CkptMeta) == 16, "CkptMeta layout");

// Geometry of the paged pool and of one head record.
struct PoolView {
    uint8_t *base;
    int64_t page_bytes;
    int32_t num_pages;
    int32_t pages_per_object;
    int64_t rec_bytes;   // bytes of one head record (multiple of 256)
    int32_t page_shift;  // log2(page_bytes) when that is a power of two, else -1
    uint32_t page_magic; // ceil(2^32 / page_bytes) for other sizes below 4 GiB, else 0
};

struct PrefillArgs {
    int32_t H, d, dtype, nseq;
    int64_t T_tot;                // rows of the packed token arrays
    const void *q, *k, *v, *alpha, *beta;
    const float *conv_w;
    void *o;
    PoolView pool;
    const SeqMeta *seqs;
    const CkptMeta *ckpts;
    const int32_t *pages;
    int32_t *status;
};

// Split prefill (bf16, d = 128): a parallel chunk preparation writes one operand image per
// (chunk, head) item, a sequential chain consumes the images in chunk order.  The chunks of
// every chain are processed in waves (wave w = local chunks [wave_c0[w], wave_c0[w + 1]));
// wave w's images live in slot w % 2 of the image buffer.
constexpr int64_t kImageBytes = 82432;   // [-WK' Gamma_C | q gamma_r] 32 KiB | [P^T | Kb] 24 KiB | V 16 KiB |
                                         // T 8 KiB | gamma_C 512 B

struct SplitItem {
    int32_t seq;   // sequence
    int32_t lc;    // chunk index within the sequence's chain
    int32_t row0;  // packed-token row of the chunk's first position (below the sequence's first
                   // row for a chunk that starts before start_pos)
    int32_t ckpt;  // index in the checkpoint table of the checkpoint at the chunk's end, or -1
};

struct SplitArgs {
    PrefillArgs p;
    const SplitItem *items;        // every wave's items, wave after wave
    const int32_t *wave_seq_off;   // [nwaves][nseq]: index in its wave of item (s, wave_c0[w]), -1 if none
    uint8_t *images;               // [2 slots][slot_items][H][kImageBytes]
    int64_t slot_items;            // items one slot holds
    float *state_scr;              // [nseq][H][d][d] state handed from one wave to the next
    uint8_t *win_scr;              // [nseq][H][3][3d] bf16 final conv window
    int32_t nwaves;
};

// Host-side wave plan of a split prefill call.
struct SplitPlan {
    int32_t nwaves = 0;
    int64_t slot_items = 0;
    std::vector<int32_t> wave_c0;        // [nwaves + 1] first local chunk of every wave
    std::vector<SplitItem> items;
    std::vector<int32_t> wave_begin;     // [nwaves + 1] offsets into items
    std::vector<int32_t> wave_seq_off;   // [nwaves * nseq]
};

struct DecodeArgs {
    int32_t H, d, dtype, B;
    const void *q, *k, *v, *alpha, *beta;
    const float *conv_w;
    void *o;
    PoolView pool;
    const int32_t *state_pages;   // [B * P] read
    const int32_t *dst_pages;     // [B * P] written (== state_pages for the in-place step)
    int32_t *status;
};

// Speculative verify: K draft tokens per request applied one after another; the state after
// draft token j of request b goes to its own object.
struct VerifyArgs {
    int32_t H, d, dtype, B, K;
    const void *q, *k, *v, *alpha;   // [K][B][H][d] (draft-token major)
    const void *beta;                // [K][B][H]
    const float *conv_w;
    void *o;                         // [K][B][H][d]
    PoolView pool;
    const int32_t *src_pages;        // [B * P] read only
    const int32_t *inter_pages;      // [K][B][P] written
    int32_t *status;
};

struct CopyArgs {
    int32_t n;                    // objects
    int64_t object_bytes;
    PoolView pool;
    const int32_t *src_pages;     // [n * P]
    const int32_t *dst_pages;     // [n * P]
    int32_t *status;
};

// Object copy between the paged pool and device-mapped host memory (object i at host +
// i * object_bytes).
struct HostCopyArgs {
    int32_t n;
    int64_t object_bytes;
    PoolView pool;
    const int32_t *pages;         // [n * P]
    uint8_t *host;                // device address of the host buffer
    int32_t to_host;              // 1: pool -> host (offload), 0: host -> pool (prefetch)
    int32_t *status;
};

// INT8 checkpoint conversion between full-precision objects and INT8 checkpoint objects.
struct Q8Args {
    int32_t n, H, d, dtype;
    PoolView full, q8;            // geometry of the full-precision and of the INT8 objects
    const int32_t *full_pages;    // [n * full.pages_per_object]
    const int32_t *q8_pages;      // [n * q8.pages_per_object]
    int32_t *status;
};

// Kernel launchers (defined in the .cu files).
cudaError_t launch_prefill_split(const SplitArgs &a, const SplitPlan &plan, cudaStream_t s);
cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
bool prefill_tc_supported(const PrefillArgs &a);
// Prefill dispatch: the tensor-core kernel for bf16 with d = 128, the fp32 CUDA-core kernel
// otherwise (fp32 inputs need fp32 arithmetic to meet their tolerance).
inline cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
    return prefill_tc_supported(a) ? launch_prefill_tc(a, s) : launch_prefill_simt(a, s);
}
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
// Fused verify kernel (bf16, d = 128, pages of at least 64 KiB, K <= kVerifyFusedMaxK): every
// source record is read once and the state stays on chip across the K draft tokens.
constexpr int kVerifyFusedMaxK = 8;
bool verify_fused_supported(const VerifyArgs &a);
cudaError_t launch_verify_fused(const VerifyArgs &a, cudaStream_t s);
cudaError_t launch_copy_objects(const CopyArgs &a, cudaStream_t s);
cudaError_t launch_host_copy(const HostCopyArgs &a, cudaStream_t s);
cudaError_t launch_ckpt_quantize(const Q8Args &a, cudaStream_t s);
cudaError_t launch_ckpt_dequantize(const Q8Args &a, cudaStream_t s);

}  // namespace kda
