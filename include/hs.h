/*
 * hs.h -- C ABI of the hierarchical KV cache resolver for top-k sparse-attention decoding (GB300, sm_103a).
 *
 * The method is the per-layer selection resolution of "HiSparse: Scaling Sparse-Attention Decoding with
 * Hierarchical KV Cache Management" (Abstract): every request keeps its whole KV history in host memory and a small
 * GPU cache of fixed size; for each layer, one kernel inside the decode step's CUDA graph looks the layer's top-k
 * selections up in that cache, makes room by least-recently-used replacement and fetches what is missing from host
 * memory; where layers share one selection, the next layer is prefetched exactly. By the "HiSparse" knowledge card
 * (Timeline) only missing rows that the top-k actually selects are brought over, and by the "Hybrid HiSparse" card
 * (Timeline) the single-pass kernel can be captured in a CUDA graph.
 *
 * Cache instance. One request-layer (layer l, request b) owns `slots` hot rows of `row_bytes` bytes and three
 * int32 arrays in device memory: tok2slot[ctx] (slot holding token t, or -1), slot_tok[slots] (token in slot v,
 * or -1) and slot_stamp[slots] (decode step of the slot's last hit or fill, 0 = never used).
 *
 * Policy of one resolve call at decode step s, for the selection S = topk_idx[b][0..k):
 *   - a negative entry is padding (its out_slot is -1, it touches nothing);
 *   - if S holds a token >= ctx or a token twice, the row is rejected: its out_slots are all -1, nothing
 *     changes, and the sticky device error word gets HS_DEVERR_RANGE / HS_DEVERR_DUP;
 *   - hits (tok2slot[t] >= 0) take stamp s;
 *   - misses, in ascending token order, take the victims: the slots not hit by this call with the smallest
 *     (stamp, slot index), in that order; the victim's old token is unmapped, the miss token mapped, the
 *     slot stamped s, and the token's row copied from the host pool into the slot;
 *   - out_slots[b][i] = slot now holding topk_idx[b][i], in input order.
 *
 * Ownership: every byte of host and device memory is the caller's. The library allocates nothing on the hot
 * path; it keeps only the small opaque hs_pool struct on the host.
 *
 * Errors: functions return HS_OK (0) or a negative HS_ERR_* code. Argument errors never launch anything. Input
 * errors that only the device can see (a bad token) never trap: they set bits of the device error word, read
 * with hs_get_error.
 *
 * Streams and graphs: hs_pool_create, hs_pool_reset, hs_step_begin and the resolve calls (hs_resolve, hs_prefetch,
 * their _ids forms, hs_resolve_shared, hs_resolve_tiered) only enqueue work on the given stream (no host
 * synchronisation) and can be captured into a CUDA graph. The kernels use
 * programmatic dependent launch: each waits for the preceding kernel in its stream before touching memory.
 * Pointers, batch and k are baked into a captured graph; refill topk_idx in place between replays.
 * The hs_get_* readers synchronise the device. No function is thread-safe on the same pool.
 *
 * Where the per-call arrays may live: topk_idx, req_ids, resident_row and out_slots may be device memory or page-locked
 * host memory mapped into the device's address space (hs_host_alloc, or cudaHostAlloc with
 * cudaHostAllocMapped; pass the device-side address, which equals the host address under unified addressing,
 * as on GB300). The kernels then read the selection and write the slots over the host link (NVLink-C2C)
 * themselves, with no separate copy; index loads always fetch afresh, so the host may rewrite a selection
 * buffer between calls. Host-side writes must be complete before the call is enqueued, and out_slots in host
 * memory may be read once the stream has been synchronised. Metadata, hot buffer and pool stay as described
 * in hs_pool_desc.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers; pass 0 for the legacy default stream. */
typedef struct CUstream_st *hs_stream_t;

typedef struct hs_pool hs_pool;

/* Return codes. */
#define HS_OK 0
#define HS_ERR_INVALID_ARG (-1) /* bad pointer, size, alignment, layer, batch or k; nothing launched */
#define HS_ERR_CUDA (-2)        /* a CUDA runtime call or launch failed */
#define HS_ERR_NOT_MAPPED (-3)  /* host_pool is not page-locked, device-mapped memory */
#define HS_ERR_NO_MEMORY (-4)   /* host struct allocation failed */
#define HS_ERR_UNSUPPORTED (-5) /* geometry needs more shared memory per block than the device offers */
#define HS_ERR_TOO_LARGE (-6)   /* request larger than the fixed device scratch of hs_probe_link_static */

/* Bits of the sticky device error word. */
#define HS_DEVERR_RANGE 1 /* a selected token was >= ctx */
#define HS_DEVERR_DUP 2   /* a token appeared twice in one selection row */
#define HS_DEVERR_STATE 4 /* metadata found inconsistent (never set by correct use) */
#define HS_DEVERR_TIMEOUT 8 /* a kernel's bounded wait ran out and it stopped early (never set by correct use) */

/*
 * Geometry and memory of a pool of layers x max_batch request-layers.
 *   layers, max_batch, ctx, slots, topk_max: >= 1; topk_max <= slots <= 65535 (k selections never exceed the
 *     fixed-size cache, "HiSparse" paper, Abstract: the GPU cache bounds the decode footprint).
 *   row_bytes: bytes of one KV row (or page); > 0 and a multiple of 16.
 *   host_pool: host rows of request b, layer l, token t at
 *       host_pool + l*host_layer_stride + b*host_req_stride + t*row_bytes.
 *     Must be page-locked and mapped into the device address space (cudaHostAlloc with cudaHostAllocMapped,
 *     or hs_host_alloc) and 16-byte aligned. May be NULL when noio_src is given.
 *   host_layer_stride: bytes between layers; 0 lets every layer read one shared pool, and a stride smaller than
 *     a layer makes the layers' rows overlap (for benchmarks whose full history does not fit in host memory: a
 *     stride of a few rows gives layers with the same selection different rows to fetch). Multiple of 16, >= 0.
 *     Scattered rows arrive more slowly the more host memory a step's layers spread them over (the host's side
 *     of the fetch, most likely address translation, bounds them, not the link), so shared or overlapping pools
 *     measure an optimistic step.
 *   host_req_stride: bytes between requests; 0 means ctx*row_bytes. Multiple of 16.
 *   hot_buf: device memory [layers][max_batch][slots][row_bytes], 16-byte aligned. Not initialised here.
 *   meta: device memory of hs_meta_bytes(desc) bytes, 256-byte aligned, holding the metadata arrays, the step
 *     counter, the counters and the error word. Initialised by hs_pool_create.
 *   noio_src: optional device copy of the row source with the same strides. When non-NULL, misses are fetched
 *     from it instead of the host pool ("no-IO" mode, which isolates the cost of resolution from host IO,
 *     "HiSparse" paper, Abstract: the no-IO oracle).
 */
typedef struct {
  int32_t layers;
  int32_t max_batch;
  int32_t ctx;
  int32_t slots;
  int32_t topk_max;
  int32_t row_bytes;
  const void *host_pool;
  int64_t host_layer_stride;
  int64_t host_req_stride;
  void *hot_buf;
  void *meta;
  const void *noio_src;
} hs_pool_desc;

/* Byte offsets of the arrays inside `meta` (for inspection and checkpointing; the layout is stable):
 *   step: int32; error: int32 (the next int32 is the completion count of hs_step_begin_fused);
 *   counters: uint64 [layers][4] = (hits, misses, evictions, bytes fetched);
 *   tok2slot: int32 [layers][max_batch][ctx]; slot_tok, slot_stamp: int32 [layers][max_batch][slots]. */
typedef struct {
  size_t step;
  size_t error;
  size_t counters;
  size_t tok2slot;
  size_t slot_tok;
  size_t slot_stamp;
  size_t total;
} hs_meta_layout;

/* Bytes of device metadata a descriptor needs (0 if the geometry is invalid). */
size_t hs_meta_bytes(const hs_pool_desc *desc);

/* Fill *out with the metadata layout of a descriptor. HS_ERR_INVALID_ARG on a bad geometry. */
int hs_get_meta_layout(const hs_pool_desc *desc, hs_meta_layout *out);

/*
 * Validate the descriptor, bind the pool to the current device, and enqueue on `stream` the initialisation of
 * the metadata: every cache empty (tok2slot = slot_tok = -1, stamps 0), step 0, counters and error word 0.
 * *out receives the opaque handle (host memory owned by the library until hs_pool_destroy).
 * Basis: the two tiers of the HiSparse paper (Abstract) -- the full KV history in host memory and a cache of fixed
 * size on the GPU -- bound together with the per-request maps that the resolution keeps.
 */
int hs_pool_create(const hs_pool_desc *desc, hs_stream_t stream, hs_pool **out);

/* Enqueue the same initialisation again (every cache emptied, step and counters back to 0). Capturable. */
int hs_pool_reset(hs_pool *pool, hs_stream_t stream);

/* Enqueue "step += 1" on the device step counter; call once per decode step before that step's resolves.
 * Stamps are decode step numbers, so every layer resolved in one step stamps with the same value. Basis: the
 * paper's least-recently-used replacement (Abstract) read with the decode step as the unit of recency, which makes
 * a prefetch and the resolve that follows it in the same step stamp alike; the increment is a kernel so that it
 * sits inside the step's CUDA graph ("Hybrid HiSparse" knowledge card, Timeline: graph-capturable). */
int hs_step_begin(hs_pool *pool, hs_stream_t stream);

/*
 * The same step increment without a launch of its own: it is carried by the next hs_resolve, hs_prefetch,
 * hs_resolve_shared or hs_resolve_tiered call made on this pool from the host (in host call order, which is also
 * the order in which a CUDA graph captures them). That call's kernel resolves at the advanced step and its last CTA
 * stores the new step value, using the third 32-bit word of the metadata header as a completion count (left at 0),
 * so a steady decode step of one layer is one launch. Valid only when no other call on the pool runs concurrently
 * with that one (a prefetch on another stream, for instance, would read the step while it changes): pipelines
 * with hs_prefetch keep hs_step_begin. Calls made twice add up; hs_pool_reset drops pending increments. Enqueues
 * nothing; HS_ERR_INVALID_ARG for a null pool. Basis: as hs_step_begin.
 */
int hs_step_begin_fused(hs_pool *pool);

/*
 * Resolve one layer's selections for requests 0..batch-1 (batch row b is pool request b) at the current step:
 * hit test, LRU victim choice, metadata update and the fetch of every missing row into its hot slot, in one
 * kernel ("HiSparse" paper, Abstract). topk_idx: int32 [batch][k], row-major; out_slots: int32 [batch][k],
 * written in input order (device or mapped host memory, see above). 1 <= batch <= max_batch,
 * 1 <= k <= topk_max; batch == 0 or k == 0 is a no-op. Enqueued on `stream`.
 */
int hs_resolve(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *topk_idx, int32_t k,
               int32_t *out_slots, hs_stream_t stream);

/*
 * Exact layer-wise prefetch for models whose layers share one selection ("HiSparse" paper, Abstract): the same
 * resolution as hs_resolve for `layer` at the current step, without writing out_slots. A later hs_resolve of
 * the same layer and selection in the same step finds every token resident, re-stamps the hits with the same
 * step value and only emits the slots, so prefetch + resolve leaves exactly the state of resolve alone. Run it
 * on a second stream; calls on different layers touch disjoint state.
 */
int hs_prefetch(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *topk_idx, int32_t k,
                hs_stream_t stream);

/*
 * hs_resolve and hs_prefetch with a request-id indirection: batch row b (row b of topk_idx and out_slots) is
 * resolved against pool request req_ids[b] instead of request b, so a serving engine whose batch rows are not its
 * cache slots passes its mapping instead of permuting the pool. Basis: the paper keeps one cache per request
 * (Abstract); which request a batch row belongs to is the engine's, and the plain reading is a per-row request id.
 *   req_ids: int32 [batch], device or mapped host memory, read once per call; every id in 0 .. max_batch-1 and
 *     distinct within a call (two rows with one id would update that request's metadata concurrently: not
 *     checked, like the distinct tokens of a row). A row whose id is out of range is rejected whole before any of
 *     the pool is read: its out_slots are -1 and the error word gets HS_DEVERR_RANGE; the other rows proceed.
 *   Everything else as hs_resolve / hs_prefetch (the per-request host pool rows and hot-buffer slots are those of
 *   request req_ids[b]); HS_ERR_INVALID_ARG also for a null req_ids.
 */
int hs_resolve_ids(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *req_ids, const int32_t *topk_idx,
                   int32_t k, int32_t *out_slots, hs_stream_t stream);
int hs_prefetch_ids(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *req_ids, const int32_t *topk_idx,
                    int32_t k, hs_stream_t stream);

/*
 * One resolve for `nlayers` consecutive layers layer0 .. layer0+nlayers-1 that share one selection per request
 * (the models for which the HiSparse paper, Abstract, prefetches layer by layer). Layers that are always resolved
 * together with the same selection hold identical metadata, so the victims are worked out once, from layer0, and
 * every layer gets the same metadata update and its own rows (from its own part of the host pool) copied into its
 * own hot buffer. The result -- state, counters, out_slots -- is exactly that of hs_resolve on each layer in turn.
 * Precondition: the nlayers layers hold identical metadata (true when they have only ever been resolved through
 * this call, or with identical selections). Arguments as hs_resolve; 1 <= nlayers, layer0 + nlayers <= layers.
 */
int hs_resolve_shared(hs_pool *pool, int32_t layer0, int32_t nlayers, int32_t batch, const int32_t *topk_idx,
                      int32_t k, int32_t *out_slots, hs_stream_t stream);

/*
 * Three-tier variant ("Hybrid HiSparse" knowledge card, Timeline: resident, hot and missing rows resolved in one
 * fused pass; hot pages come from ordinary KV blocks of the same memory pool). resident_row: int32, for request
 * b at resident_row + b*resident_stride (resident_stride >= ctx; normally device memory), the row of each token
 * still held in the ordinary HBM KV pool (0 <= row <= 2^31 - 3), or -1. A selected token that is not in the hot
 * buffer but is resident there is served in place: it takes no slot, refreshes no stamp, is fetched from nowhere,
 * counts as a hit, and its out_slot is -2 - row. A hot-buffer hit takes precedence. Everything else is as
 * hs_resolve.
 */
int hs_resolve_tiered(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *topk_idx, int32_t k,
                      const int32_t *resident_row, int64_t resident_stride, int32_t *out_slots,
                      hs_stream_t stream);

/*
 * The read a sparse-attention kernel makes after a resolve: for every request b < batch and entry i < k, copy hot
 * row out_slots[b][i] of `layer` to dst + (b*k + i)*row_bytes (a zero row for -1). dst: device memory of
 * batch*k*row_bytes bytes, 16-byte aligned. Enqueued on `stream`. Together with hs_gather_history it shows that
 * placement changes nothing the attention reads ("HiSparse" paper, Abstract: model outputs are unchanged).
 */
int hs_gather(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *out_slots, int32_t k, void *dst,
              hs_stream_t stream);

/* The same read from the full history: dst row (b, i) = host-pool row topk_idx[b][i] of `layer` (from the no-IO
 * source when the pool has one; a zero row for an index < 0 or >= ctx). */
int hs_gather_history(hs_pool *pool, int32_t layer, int32_t batch, const int32_t *topk_idx, int32_t k, void *dst,
                      hs_stream_t stream);

/*
 * Consumer: sparse MLA decode attention over the rows a resolve selected, on the tensor cores (the read that the
 * hot buffer exists for: "HiSparse" paper, Abstract, the model's outputs do not change; the "Hybrid HiSparse" card
 * builds on Sparse MLA). Absorbed multi-head latent attention, one decode step: every row is 576 bf16 values (the
 * 512-value latent, then the 64-value rotary key), so the pool's row_bytes must be 1152 (else
 * HS_ERR_UNSUPPORTED). For request b < batch and head h < 128, over the valid entries i of its slot list:
 *     s[h][i] = sm_scale * dot(q[b][h][0:576], row_i),
 *     out[b][h][0:512] = sum_i softmax_i(s[h]) * row_i[0:512],   lse[b][h] = ln sum_i exp(s[h][i]).
 * out_slots [batch][k] as a resolve wrote it (device or mapped host memory): an entry >= 0 names hot slot
 * `entry` of `layer`; an entry <= -2 names row -2 - entry of resident_rows (device, 1152-byte rows, count rows;
 * NULL for none), as hs_resolve_tiered writes them; -1 and anything else is padding. q: device bf16
 * [batch][128][576], 16-byte aligned; out: device fp32 [batch][128][512], 16-byte aligned; lse: device fp32
 * [batch][128]. With no valid entry a head's output is zero and its lse -inf. P is rounded to bf16 before the
 * value product and the normaliser sums the rounded weights; scores and outputs accumulate in fp32. When the
 * device holds a cluster of four CTAs for every request at once, each request's keys are split in two halves
 * whose softmaxes are merged at the end, with `out` holding the halves' partial outputs in between: out must not
 * overlap q, the slot list or the rows. Results are deterministic for a given batch size; a split and
 * an unsplit launch round differently, within the same error bound. Enqueued on `stream`; batch == 0 or k == 0
 * is a no-op.
 */
int hs_mla_decode(hs_pool *pool, int32_t layer, int32_t batch, const void *q, const int32_t *out_slots, int32_t k,
                  const void *resident_rows, int64_t resident_count, float sm_scale, float *out, float *lse,
                  hs_stream_t stream);

/* The same attention read from the full history, for comparison: entry i of topk_idx names token i of request
 * b's rows in the pool's row source (the no-IO copy when the pool has one, else the host pool); indices < 0 or
 * >= ctx are padding. Equal rows in the same order give bit-identical out and lse. */
int hs_mla_decode_history(hs_pool *pool, int32_t layer, int32_t batch, const void *q, const int32_t *topk_idx,
                          int32_t k, float sm_scale, float *out, float *lse, hs_stream_t stream);

/*
 * Test hook of the attention consumer (not for production use; process-wide settings, not thread-safe). It lets a
 * test exercise failure detection without faulting the GPU: every wait inside the kernel is bounded, and on running
 * out it stops every role, frees its tensor memory, returns and sets HS_DEVERR_TIMEOUT.
 *   wait_limit: polling rounds after which a wait of the kernel's roles gives up (0 restores the default, 2^20).
 *   stall != 0: the tensor-core issuer of every CTA first waits on a barrier that nothing completes, so that wait
 *     runs out before any tensor-core work or row copy of the kernel is issued, and the abort path runs with
 *     nothing in flight. 0 restores normal operation.
 *   split_max_batch: if non-NULL, receives the largest batch for which hs_mla_decode splits a request's keys over
 *     two CTA pairs on the current device (larger batches run one pair per request).
 * Applies to the hs_mla_decode / hs_mla_decode_history calls made after it.
 */
int hs_debug_attention(uint32_t wait_limit, int32_t stall, int32_t *split_max_batch);

/* Synchronise the device, then read the sticky device error word into *out (HS_DEVERR_* bits); clear it when
 * `clear` is non-zero. Basis: the pages say nothing about bad selections; the reading taken here is that a kernel
 * inside a decode graph must never trap, so a row it cannot resolve is rejected and reported here instead. */
int hs_get_error(hs_pool *pool, int32_t *out, int32_t clear);

/* Synchronise the device, then read layer `layer`'s counters: out[0..3] = hits, misses, evictions, bytes.
 * Every call counts: a resolve that follows a prefetch of the same selection adds its k lookups as hits. Basis:
 * the paper measures the cost of the method as the host-to-device traffic of misses (Abstract); these are the
 * counts that traffic follows from. */
int hs_get_counters(hs_pool *pool, int32_t layer, uint64_t out[4]);

/* Release the opaque handle. Caller memory is untouched. Basis: as hs_pool_create; all memory stays the
 * caller's, so the library only frees its own small host struct. */
int hs_pool_destroy(hs_pool *pool);

/* Page-locked, device-mapped, portable host allocation for a host pool (not for the hot path). */
int hs_host_alloc(size_t bytes, void **out);
int hs_host_free(void *ptr);

/*
 * Measure the host link this pool fetches over (not for the hot path; synchronises and creates two events).
 * Reads `bytes` of the mapped host buffer `host` with the same 16-byte SM loads the resolve kernel uses
 * (zero-copy, all SMs), and copies them with cudaMemcpyAsync into the device buffer `dev` (>= bytes), each
 * `iters` times after one warm-up; reports the best of each in GB/s (1e9 bytes/s). bytes: multiple of 16.
 */
int hs_probe_link(const void *host, void *dev, size_t bytes, int32_t iters, hs_stream_t stream,
                  double *zero_copy_gbs, double *memcpy_gbs);

/*
 * Measure the fixed cost under a resolve (not for the hot path): enqueue a kernel that does nothing but wait for its
 * predecessor and release its dependents, launched with exactly the configuration that hs_resolve (nlayers == 1) or
 * hs_resolve_shared would use for this layer range, batch and k: grid, cluster size, dynamic shared memory and
 * programmatic dependent launch. A decode step made of these launches in place of the resolves times the floor that
 * launching alone puts under the step. Argument checks as hs_resolve_shared; touches no memory; capturable.
 */
int hs_probe_launch(hs_pool *pool, int32_t layer, int32_t nlayers, int32_t batch, int32_t k, hs_stream_t stream);

/*
 * The link probe for callers that cannot allocate device memory. hs_probe_link needs a device buffer of `bytes`
 * that serves only as scratch (the copy's destination, the read kernel's sink). A caller that links this library
 * without a device allocator of its own -- plain C code that has only the page-locked host memory of hs_host_alloc,
 * or a component whose framework hands out no scratch -- cannot provide it. This entry point allocates nothing:
 * its scratch is a fixed 16 MiB array in the library's device module (plus 256 bytes of clock stamps), which every
 * GPU that loads the library holds until the process exits. The paper has no counterpart; it is plumbing.
 *   host: mapped page-locked host memory as for hs_probe_link; bytes: a multiple of 16, 16 .. 16 MiB, else
 *   HS_ERR_TOO_LARGE (nothing is launched); iters >= 1. Same measurement as hs_probe_link (best of `iters` after one
 *   warm-up, GB/s = 1e9 bytes/s), timed by device clock stamps instead of events.
 * The first call on a device looks up the scratch's device address (cudaGetSymbolAddress) and keeps it; that call
 * synchronises, like every call. Every call shares the one scratch array, which keeps whatever the last call left
 * there (nothing in it has to start at zero): calls that overlap on the GPU -- two streams, or two host threads --
 * race on it.
 */
int hs_probe_link_static(const void *host, size_t bytes, int32_t iters, hs_stream_t stream, double *zero_copy_gbs,
                         double *memcpy_gbs);

/* Static text for an HS_ERR_* code. */
const char *hs_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
