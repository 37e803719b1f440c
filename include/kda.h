/*
 * kda.h — C ABI of the KDA state library (libkda.so) for one GB300 GPU (sm_103a).
 *
 * The library computes the Kimi Delta Attention (KDA) state path:
 *   - a chunked varlen prefill that reads q, k, v, alpha, beta, applies the width-4 causal
 *     depthwise conv to q | k | v, runs the recurrence
 *         S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t
 *     (decay first, then the delta-rule write, then the read: "Lesson 01 · Architecture
 *     map", §两种 Attention，两种状态), writes o, streams checkpoints of (S, conv window) at
 *     a sparse subset of 512-token hash-block ends into a paged pool ("Cache de préfixe
 *     hybride KDA–MLA", §La solution and §Le fonctionnement du prefill) and writes the
 *     final state to the sequence's private (active) object;
 *   - resume from any checkpoint: copy it into the private object, then prefill with
 *     has_init = 1 (same page, §Les checkpoints sont en lecture seule);
 *   - a batched single-token decode step that gathers each request's state through a page
 *     table and updates it in place ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제",
 *     §0x08 8.2.2: conv state and recurrent state handed to a fused decode kernel).
 *
 * Conventions
 * -----------
 * - Every function returns a kda_status (int); functions that return a count return it as
 *   a non-negative value and errors as negative kda_status values.
 * - dtype: KDA_F32 or KDA_BF16; it is the type of q, k, v, alpha, beta, o and of the conv
 *   window stored in records.  The recurrent state is always fp32.  conv_w is always fp32.
 * - "device" pointers are CUDA device addresses on the current device; "host" pointers are
 *   ordinary host memory that is read (or written) before the call returns.
 * - The caller owns every device buffer (inputs, outputs, the pool base, page tables, the
 *   workspace and the int32 device status word).  The library owns only the host-side pool
 *   metadata behind the opaque kda_pool (free set, reference counts) and a few pinned host
 *   staging buffers that carry call metadata to the workspace.
 * - GPU work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *   stream).  Buffers handed to a call must stay alive until that work completes.
 * - Nothing aborts or traps.  Host-side argument errors return KDA_EINVAL / KDA_ENOPAGES /
 *   KDA_EREF before anything is enqueued.  Kernels check page ids and metadata and, on a bad
 *   value, skip the access and set a bit in *status_dev; kda_sync_status reports it as
 *   KDA_EDEVICE.  CUDA launch errors return KDA_ECUDA.
 * - A kda_pool may be used from one host thread at a time.
 *
 * Paged state layout (bit-exact)
 * ------------------------------
 * One page byte size for the whole pool.  A head record is S as fp32 row-major [d][d]
 * (row i = key channel i, column j = value channel j), then the conv window [3][3d] in
 * dtype (oldest raw token first, channels q | k | v), zero-padded to a multiple of 256
 * bytes.  An object is the H head records of one sequence, one after another in head order
 * (heads stored contiguously: "Cache de préfixe hybride KDA–MLA", §La mise en page
 * unifiée).  Logical byte x of an object lives in page list[x / page_bytes] at byte
 * x % page_bytes of that page; the page lists are int32 [P] with P = kda_object_pages().
 */
#ifndef KDA_H
#define KDA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status_code {
    KDA_OK = 0,
    KDA_EINVAL = -1,    /* bad argument, shape, dtype, position or size */
    KDA_ENOPAGES = -2,  /* pool exhausted: nothing was allocated */
    KDA_EREF = -3,      /* reference-count misuse (freeing a free page, claiming a used one) */
    KDA_ECUDA = -4,     /* CUDA launch / runtime error */
    KDA_EDEVICE = -5    /* a kernel found a bad page id, bad metadata or an out-of-range decay
                           (see kda_sync_status) */
} kda_status_code;

typedef enum kda_dtype { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Device status bits set by kernels (reported through kda_sync_status). */
#define KDA_DEV_BAD_PAGE 1   /* a page id outside [0, num_pages) was met; access skipped */
#define KDA_DEV_BAD_META 2   /* inconsistent metadata in the workspace; work skipped */
#define KDA_DEV_TIMEOUT 4    /* an internal pipeline wait gave up; that sequence is incomplete */
#define KDA_DEV_RANGE 8      /* prefill: a chunk's decay product fell below the supported range
                                (see alpha in kda_prefill_varlen); that sequence's results are undefined */

typedef struct kda_pool kda_pool;

/* ---------------------------------------------------------------- sizes --------------- */

/* Bytes of one head record for head dimension d (64 or 128) and dtype; KDA_EINVAL if bad. */
int64_t kda_record_bytes(int32_t d, int32_t dtype);

/* Bytes of one object (H records).  KDA_EINVAL if bad. */
int64_t kda_object_bytes(int32_t H, int32_t d, int32_t dtype);

/* Pages per object in this pool: ceil(kda_object_bytes / page_bytes).  KDA_EINVAL if bad. */
int32_t kda_object_pages(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype);

/* ---------------------------------------------------------------- pool ---------------- */
/* One refcounted page allocator for every state object ("Cache de préfixe hybride
 * KDA–MLA", §La mise en page unifiée: one allocation / reference-count / eviction path for
 * all page kinds).  Device memory for the pages is the caller's: num_pages * page_bytes
 * bytes at `pool_base`, passed to each GPU call. */

/* page_bytes must be a positive multiple of 256; num_pages > 0.  *out receives the pool. */
int kda_pool_create(int64_t page_bytes, int32_t num_pages, kda_pool **out);
/* Frees the pool's host metadata and its pinned staging buffers, first waiting for any
 * upload still reading them; the caller's device pages are untouched.  KDA_EINVAL for NULL. */
int kda_pool_destroy(kda_pool *pool);
/* The page size in bytes, the number of pages, and the number of free pages (reference count
 * 0).  KDA_EINVAL for NULL. */
int64_t kda_pool_page_bytes(const kda_pool *pool);
int32_t kda_pool_num_pages(const kda_pool *pool);
int32_t kda_pool_free_count(const kda_pool *pool);

/* Allocate n pages, lowest free id first, each with refcount 1; ids written to out_ids[n].
 * KDA_ENOPAGES (nothing allocated) if fewer than n pages are free. */
int kda_page_alloc(kda_pool *pool, int32_t n, int32_t *out_ids);

/* Take the n given free pages (refcount 0 -> 1), e.g. to follow a caller's page table.
 * KDA_EREF if any is in use or repeated, KDA_EINVAL if out of range; all or nothing. */
int kda_page_claim(kda_pool *pool, int32_t n, const int32_t *ids);

/* Pin (refcount + 1) n pages that are in use; KDA_EREF if one is free.  All or nothing.
 * Pinning every hit page before any allocation is the first concurrency rule of "Cache de
 * préfixe hybride KDA–MLA", §La cohérence sous ordonnancement concurrent. */
int kda_page_incref(kda_pool *pool, int32_t n, const int32_t *ids);

/* Unpin n pages; a page is free again at refcount 0.  KDA_EREF if a count would go below
 * zero (repeated ids count once per occurrence).  All or nothing. */
int kda_page_decref(kda_pool *pool, int32_t n, const int32_t *ids);

/* Refcount of page id, or KDA_EINVAL if out of range. */
int32_t kda_page_refcount(const kda_pool *pool, int32_t id);

/* ---------------------------------------------------------------- policy -------------- */

/* Checkpoint positions of one forward over absolute positions [start, end): every p with
 * p % (hash_block * stride) == 0 and start < p <= end, plus floor(end / hash_block) *
 * hash_block when include_last != 0 and it is > start ("Cache de préfixe hybride KDA–MLA",
 * §La solution: a sparse subset of hash-block ends; §Le fonctionnement du prefill: persist
 * the last hash-aligned position processed).  Writes up to cap ascending positions to out
 * and returns the total count (which may exceed cap), or KDA_EINVAL. */
int32_t kda_ckpt_positions(int64_t start, int64_t end, int32_t hash_block, int32_t stride,
                           int32_t include_last, int64_t *out, int32_t cap);

/* Plan the checkpoints of one prefill call and allocate their objects.  Sequence s covers
 * absolute positions [start_pos[s], start_pos[s] + cu_seqlens[s+1] - cu_seqlens[s]).
 * Checkpoints are listed in (sequence ascending, position ascending) order and each gets P
 * fresh pages, lowest free first, refcount 1 (new checkpoints go to fresh slots: "Cache de
 * préfixe hybride KDA–MLA", §Les checkpoints sont en lecture seule).  Outputs (host):
 * *out_n, out_seq[cap], out_pos[cap], out_pages[cap * P].  KDA_EINVAL if more than cap
 * checkpoints would result; KDA_ENOPAGES if the pool cannot hold them (nothing allocated).
 * hash_block must be a positive multiple of 64. */
int kda_ckpt_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                  const int32_t *cu_seqlens, const int64_t *start_pos, int32_t hash_block,
                  int32_t stride, int32_t include_last, int32_t cap, int32_t *out_n,
                  int32_t *out_seq, int64_t *out_pos, int32_t *out_pages);

/* ---------------------------------------------------------------- prefill ------------- */

/* Workspace bytes kda_prefill_varlen needs for this batch (the same arguments as that call):
 *   H, d, dtype            heads, head dimension, token dtype
 *   nseq, cu_seqlens, start_pos   host arrays as in kda_prefill_varlen (they may be NULL when
 *                          the path for this shape needs metadata only: fp32 or d = 64)
 *   n_ckpt, pages_per_object      the checkpoint count of the call and kda_object_pages()
 * For bf16 with d = 128 the workspace also holds the chunk-operand images of the split
 * tensor-core prefill: two slots of at most ~512 MiB of images each (one image of 82,432 B per
 * (chunk, head) of a wave of chunks), plus the state handed between waves (64 KiB per
 * (sequence, head), when there is more than one wave) and the final conv windows.  Returns
 * the byte count, or KDA_EINVAL for a bad shape or inconsistent arrays. */
int64_t kda_prefill_workspace_bytes(int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                                    const int32_t *cu_seqlens, const int64_t *start_pos,
                                    int32_t n_ckpt, int32_t pages_per_object);

/* Number of kernel launches kda_prefill_varlen makes for this batch (same arguments as
 * kda_prefill_workspace_bytes; cu_seqlens / start_pos host arrays): one for fp32 or d = 64;
 * for bf16 with d = 128, two per wave of chunks (chunk preparation and chains, the
 * preparation of a wave overlapping the chains of the one before), or one when every
 * sequence is empty.
 * KDA_EINVAL for a bad shape. */
int32_t kda_prefill_kernel_launches(int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                                    const int32_t *cu_seqlens, const int64_t *start_pos);

/* The wave split of the bf16 d = 128 prefill for this batch (same arguments as
 * kda_prefill_kernel_launches): wave w covers local chunks [wave_c0[w], wave_c0[w + 1]) of
 * every sequence (local chunk 0 = the chunk holding start_pos).  Writes min(cap, W + 1) bounds
 * to the host array wave_c0 (may be NULL when cap = 0) and returns the wave count W (0 when
 * every sequence is empty, or for shapes that do not take the split path).  The split is
 * chosen by a cost model among splits whose operand images fit one workspace slot; it changes
 * speed only, never results.  KDA_EINVAL for a bad shape or inconsistent arrays. */
int32_t kda_prefill_waves(int32_t H, int32_t d, int32_t dtype, int32_t nseq, const int32_t *cu_seqlens,
                          const int64_t *start_pos, int32_t *wave_c0, int32_t cap);

/* Chunked varlen prefill (chunk = 64 tokens, chunks aligned to absolute positions).
 *   H, d, dtype      heads, head dimension (64 or 128), dtype of the token tensors
 *   nseq             number of sequences (>= 1)
 *   cu_seqlens       host int32 [nseq + 1], token offsets into the packed arrays
 *   start_pos        host int64 [nseq], absolute position of each sequence's first token
 *   has_init         host uint8 [nseq]; 1 = read the initial (S, window) from the active
 *                    object, 0 = start from zeros
 *   q, k, v, alpha   device [T_tot][H][d] dtype (q, k as given: any normalisation is the
 *                    caller's; the conv runs here)
 *                    alpha is the forget gate, in [0, 1] per key channel.  The chunked
 *                    kernels factor a chunk's decay through its running product per channel,
 *                    so the product of alpha over each 64-token chunk must stay at or above
 *                    2^-100 in every channel (a geometric-mean gate above 0.34 over a full
 *                    chunk; a gate of exactly 0 is below it).  A chunk below that sets
 *                    KDA_DEV_RANGE, and the outputs, states and checkpoints of its
 *                    (sequence, head) from that chunk on are undefined.  kda_decode_step
 *                    steps token by token and has no such limit.
 *   beta             device [T_tot][H] dtype
 *   conv_w           device fp32 [H][3d][4]; tap j multiplies raw token t-3+j
 *   o                device [T_tot][H][d] dtype, written
 *   pool_base        device base of the page pool
 *   active_pages     host int32 [nseq * P]: each sequence's private object (read when
 *                    has_init, always written with the final state and window)
 *   n_ckpt, ckpt_seq, ckpt_pos, ckpt_pages   host: the checkpoints to stream (as produced
 *                    by kda_ckpt_plan): sequence ids ascending, positions ascending within
 *                    a sequence, each position p with start < p <= end and p % 64 == 0 or
 *                    p == end; ckpt_pages [n_ckpt * P] must be allocated pages
 *   workspace        device scratch (16-byte aligned) of at least
 *                    kda_prefill_workspace_bytes() for the same batch; the call
 *                    writes metadata there (one async host-to-device copy)
 *   status_dev       device int32 status word (bits KDA_DEV_*), OR-ed by the kernel
 * The state checkpoint at p is S after tokens [0, p) with the raw tokens p-3, p-2, p-1 as
 * window, in the record layout above. */
int kda_prefill_varlen(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                       const int32_t *cu_seqlens, const int64_t *start_pos,
                       const uint8_t *has_init, const void *q, const void *k, const void *v,
                       const void *alpha, const void *beta, const float *conv_w, void *o,
                       void *pool_base, const int32_t *active_pages, int32_t n_ckpt,
                       const int32_t *ckpt_seq, const int64_t *ckpt_pos,
                       const int32_t *ckpt_pages, void *workspace, int64_t ws_bytes,
                       int32_t *status_dev, void *stream);

/* Bytes of the fixed device scratch used by kda_prefill_varlen_noalloc. */
#define KDA_NOALLOC_SCRATCH_BYTES (1 << 20)

/* Allocation-free variant of kda_prefill_varlen.  The source pages have no counterpart:
 * this is an interface convenience of this library.  It serves callers that cannot
 * allocate device memory when they call the prefill: a serving runtime that reserved all
 * of HBM for its own pool at start-up (a cudaMalloc there fails or fragments that pool),
 * or a latency-critical path where cudaMalloc / cudaFree and the device synchronisation
 * they can cause are not allowed.  Arguments and results are those of kda_prefill_varlen
 * without the workspace: the per-call metadata goes to a fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES bytes inside the library's device image, which every GPU that
 * loads the library holds until the process exits.
 *   - Metadata that does not fit (32 bytes per sequence and 16 per checkpoint, each part
 *     rounded up to 256 bytes, plus 4 * (nseq + n_ckpt) * pages_per_object bytes of page
 *     lists) returns KDA_EINVAL and enqueues nothing.
 *   - The first call on each device looks up the array's device address, with that device
 *     current; make that first call before any stream capture.
 *   - Every call reuses the one array and overwrites all of the metadata it reads, so no
 *     state carries over between calls; calls whose GPU work may overlap (different streams
 *     without ordering between them) race on it.  Calls on one stream are ordered.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine: the metadata is built
 *     in a static host buffer and sent with one cudaMemcpyAsync from that pageable buffer.
 *     A copy from pageable memory is staged by the runtime before the call returns, and it
 *     can make the host wait for work already queued on the stream. */
int kda_prefill_varlen_noalloc(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t nseq,
                               const int32_t *cu_seqlens, const int64_t *start_pos,
                               const uint8_t *has_init, const void *q, const void *k,
                               const void *v, const void *alpha, const void *beta,
                               const float *conv_w, void *o, void *pool_base,
                               const int32_t *active_pages, int32_t n_ckpt,
                               const int32_t *ckpt_seq, const int64_t *ckpt_pos,
                               const int32_t *ckpt_pages, int32_t *status_dev, void *stream);

/* ---------------------------------------------------------------- decode -------------- */

/* One decode step for B requests, one token each.  q, k, v, alpha device [B][H][d] dtype,
 * beta device [B][H] dtype, conv_w device fp32 [H][3d][4], o device [B][H][d] dtype.
 * state_pages device int32 [B * P]: the page table of each request's active object, read
 * and updated in place (S and the conv window: the window is shifted by one token).
 * Page ids outside the pool set KDA_DEV_BAD_PAGE and that (request, head) is skipped. */
int kda_decode_step(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B,
                    const void *q, const void *k, const void *v, const void *alpha,
                    const void *beta, const float *conv_w, void *o, void *pool_base,
                    const int32_t *state_pages, int32_t *status_dev, void *stream);

/* Ping-pong decode step: as kda_decode_step, but each request's state is read from its
 * source object (src_pages, device int32 [B * P]) and written, with the shifted window, to its
 * destination object (dst_pages, device int32 [B * P]).  A request whose two page lists are
 * equal is updated in place; for one whose lists differ (and do not overlap), the source
 * object is left untouched and holds the state at the request's position: a decode-interval
 * checkpoint taken without a copy, which the caller donates to the cache while the request
 * continues on the destination object ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제", §0x05
 * 5.2: decode checkpoints at a fixed interval; §0x06 6.7 and 6.8: a second slot requested at a
 * checkpoint boundary, the new state written to it, the old slot donated).  Page ids outside
 * the pool in either list set KDA_DEV_BAD_PAGE and the request is skipped. */
int kda_decode_step_pp(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B,
                       const void *q, const void *k, const void *v, const void *alpha,
                       const void *beta, const float *conv_w, void *o, void *pool_base,
                       const int32_t *src_pages, const int32_t *dst_pages, int32_t *status_dev,
                       void *stream);

/* Host plan of a ping-pong step at decode-checkpoint interval `interval`:
 *   pos           host int64 [B]: tokens each request has consumed (its state's position)
 *   active_pages  host int32 [B * P]: the requests' active objects (private: refcount 1)
 * Requests with pos > 0 and pos % interval == 0 are due: for each of them, in request order,
 * P fresh pages are allocated (lowest free first, refcount 1) as the destination object, and
 * the request index is appended to donated_out (host int32 [B]; count in *n_donated_out).
 * dst_pages_out (host int32 [B * P]) receives the destination lists: the fresh pages for due
 * requests, the active pages for the others.  After the step, each due request's old active
 * pages hold its checkpoint at position pos[r] and its new active object is the destination.
 * All or nothing: KDA_ENOPAGES allocates nothing. */
int kda_decode_pingpong_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B,
                             const int64_t *pos, int32_t interval, const int32_t *active_pages,
                             int32_t *dst_pages_out, int32_t *donated_out, int32_t *n_donated_out);

/* Speculative verify ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제", §0x06 6.4: a verify pass
 * carries intermediate-state indices next to the recurrent and conv states): K draft tokens per
 * request are applied one after another and the state after each of them is kept in its own
 * object, so that the state at any accepted length is available without recomputation.
 *
 * kda_verify_plan: allocate the K * B intermediate objects (lowest free first, refcount 1;
 * all or nothing) into inter_pages_out, host int32 [K][B][P] (object of token j of request b
 * at (j * B + b) * P). */
int kda_verify_plan(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K,
                    int32_t *inter_pages_out);

/* kda_verify_step: q, k, v, alpha [K][B][H][d] and beta [K][B][H] (device, dtype; draft token
 * major), o [K][B][H][d] written.  src_pages (device int32 [B * P]) holds each request's state
 * before the drafts and is not modified; inter_pages (device int32 [K][B][P]) receives the
 * state after draft token j.  1 <= K <= 64.  For bf16, d = 128, pages of at least 64 KiB and
 * K <= 8 it is one kernel that reads each source record once and keeps the state on chip
 * across the K tokens (traffic: one record read and K record writes per request-head);
 * otherwise it runs as K stream-ordered ping-pong decode steps (kda_decode_step_pp), token j
 * reading the object token j - 1 wrote. */
int kda_verify_step(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K,
                    const void *q, const void *k, const void *v, const void *alpha,
                    const void *beta, const float *conv_w, void *o, void *pool_base,
                    const int32_t *src_pages, const int32_t *inter_pages, int32_t *status_dev,
                    void *stream);

/* kda_verify_accept (host only): accepted[b] in [0, K] draft tokens kept for request b.  The
 * request's new active object is written to active_out (host int32 [B * P]): the source
 * object when accepted[b] == 0, else the object of token accepted[b] - 1.  Every other object
 * among the request's source and intermediates is released (decref).  Call it once the
 * stream has passed the verify step. */
int kda_verify_accept(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t B, int32_t K,
                      const int32_t *accepted, const int32_t *src_pages, const int32_t *inter_pages,
                      int32_t *active_out);

/* ---------------------------------------------------------------- checkpoints --------- */

/* Workspace bytes for a checkpoint copy of n objects. */
int64_t kda_copy_workspace_bytes(int32_t n, int32_t pages_per_object);

/* Snapshot: allocate n fresh objects (lowest free first, refcount 1), copy each source
 * object (host page lists src_pages [n * P]) into them and return their pages in
 * dst_pages_out [n * P] (host).  KDA_ENOPAGES if the pool cannot hold them. */
int kda_ckpt_write(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                   const int32_t *src_pages, int32_t *dst_pages_out, void *pool_base,
                   void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* Restore (copy-on-write): pin (incref) the checkpoint pages, then copy each checkpoint
 * object ckpt_pages [n * P] into the private object active_pages [n * P] (both host
 * lists).  The checkpoint is only read.  Release the pin with kda_ckpt_release once the
 * copy has completed on the stream. */
int kda_ckpt_restore(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                     const int32_t *ckpt_pages, const int32_t *active_pages, void *pool_base,
                     void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* Drop the pin kda_ckpt_restore took: decref the same n * P checkpoint page ids. */
int kda_ckpt_release(kda_pool *pool, int32_t n, int32_t pages_per_object,
                     const int32_t *ckpt_pages);

/* ---------------------------------------------------------------- host offload ------ */

/* Write-back offload and prefetch of checkpoints ("Infrastructure pour le RL à un million de
 * jetons", §La solution : découpler la rétention de la résidence GPU: an idle reusable prefix
 * is written to CPU DRAM only when it leaves the GPU, and prefetched before its next reuse).
 * The host buffer must be pinned and mapped into the device address space (cudaHostAlloc /
 * cudaHostRegister; pinned torch tensors qualify) and 16-byte aligned; object i occupies
 * bytes [i * B, (i + 1) * B) with B = kda_object_bytes(H, d, dtype), in the object's logical
 * byte order (the same bytes as in the pool).
 *
 * Offload: copy the n objects (pages: host int32 [n * P], allocated) to host_dst; the pages
 * stay allocated: the caller decrefs them once the stream has passed the copy (the eviction).
 * workspace: device, at least kda_copy_workspace_bytes(n, P).  A host buffer that is not
 * device-accessible returns KDA_EINVAL. */
int kda_ckpt_offload(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                     const int32_t *pages, void *host_dst, int64_t host_bytes, void *pool_base,
                     void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* Prefetch: allocate n * P fresh pages (lowest free first, refcount 1; returned in pages_out,
 * host int32 [n * P]) and copy the n host objects into them.  All or nothing. */
int kda_ckpt_prefetch(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                      const void *host_src, int64_t host_bytes, int32_t *pages_out, void *pool_base,
                      void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* ---------------------------------------------------------------- INT8 checkpoints -- */

/* INT8 compressed checkpoints ("KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제", §0x05 5.3 and
 * §0x06 6.6: checkpoints waiting in the cache may hold the recurrent state in INT8 while the
 * small conv window keeps its native precision; a hit is dequantised once into a fresh active
 * slot, so the recurrence itself never runs on quantised state).
 * INT8 head record: scale fp32 [d] | codes int8 [d][d] (row i = key channel i, column j =
 * value channel j) | window [3][3d] in dtype, zero-padded to a multiple of 256 bytes
 * (19,200 bytes at d = 128 bf16 against 67,840 for the full record); an INT8 object is the H
 * records in head order, paged like a full object.  scale_i = max_j |S[i][j]| / 127 and
 * code = round-to-nearest-even(S[i][j] / scale_i) clamped to [-127, 127], both divisions IEEE
 * fp32; a zero row has scale 0 and codes 0; dequantisation writes code * scale_i. */
int64_t kda_record_bytes_q8(int32_t d, int32_t dtype);
/* H INT8 records, and the pages of this pool they span; KDA_EINVAL for a bad shape or pool. */
int64_t kda_object_bytes_q8(int32_t H, int32_t d, int32_t dtype);
int32_t kda_object_pages_q8(const kda_pool *pool, int32_t H, int32_t d, int32_t dtype);

/* Snapshot n full objects (src_pages, host int32 [n * P], allocated) into n new INT8
 * checkpoint objects: allocates n * Pq fresh pages (lowest free first, refcount 1; Pq =
 * kda_object_pages_q8), returns them in dst_pages_out (host int32 [n * Pq]) and enqueues the
 * quantisation.  workspace: device, at least kda_copy_workspace_bytes(n, P).  On an error
 * nothing is allocated.  The pool's pages and every object must be below 4 GiB. */
int kda_ckpt_write_q8(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                      const int32_t *src_pages, int32_t *dst_pages_out, void *pool_base,
                      void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* Restore n INT8 checkpoints (ckpt_pages, host int32 [n * Pq], allocated) into n private full
 * objects (active_pages, host int32 [n * P], refcount 1, disjoint from the checkpoints): the
 * checkpoint pages are pinned (incref) for the conversion and released by
 * kda_ckpt_release(pool, n, Pq, ckpt_pages) once the stream has passed it. */
int kda_ckpt_restore_q8(kda_pool *pool, int32_t H, int32_t d, int32_t dtype, int32_t n,
                        const int32_t *ckpt_pages, const int32_t *active_pages, void *pool_base,
                        void *workspace, int64_t ws_bytes, int32_t *status_dev, void *stream);

/* ---------------------------------------------------------------- status -------------- */

/* Wait for `stream`, read and clear *status_dev.  Returns KDA_OK, KDA_EDEVICE (bits in
 * *bits_out if not NULL) or KDA_ECUDA. */
int kda_sync_status(int32_t *status_dev, void *stream, int32_t *bits_out);

/* Static description of a status code. */
const char *kda_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
