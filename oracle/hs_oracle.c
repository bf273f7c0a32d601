/*
 * CPU ORACLE for the hierarchical KV cache resolver. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may call it; the library path never does. It shares no code, header or
 * constant with the CUDA path.
 *
 * What it computes, for ONE request-layer cache instance and one call at decode step `step`: the per-layer
 * resolution of "HiSparse: Scaling Sparse-Attention Decoding with Hierarchical KV Cache Management" (Abstract, and
 * its AI Summary): every selected token is looked up in the GPU cache, the least recently used entries not
 * selected now make room, and only the selected rows that are missing come over from host memory ("HiSparse"
 * knowledge card, Timeline), written out as plain sequential steps:
 *
 *   0. Validation. A negative entry is padding. If any entry is >= ctx, or a non-negative token appears twice,
 *      the whole row is rejected: out_slots is -1 everywhere, no state changes, and an error bit is returned.
 *   1. Hit test. For every selected token t_i, slot tok2slot[t_i]; a slot >= 0 is a hit. Every hit slot gets
 *      stamp `step` and joins the set Sel of slots selected this call.
 *   2. Misses. M = the miss tokens sorted ascending; m = |M|.
 *   3. Victims (LRU replacement). Candidates are the slots not in Sel, ordered by the key (stamp, slot index)
 *      ascending; empty slots carry stamp 0 so they come first, lowest index first. V = the first m candidates.
 *   4. Assignment. For j = 0..m-1 with t = M[j], v = V[j], u = slot_tok[v]: if u >= 0 then tok2slot[u] = -1;
 *      tok2slot[t] = v, slot_tok[v] = t, stamp[v] = step, and the row_bytes bytes of host row t are copied
 *      into hot slot v.
 *   5. Output. out_slots[i] = tok2slot[t_i] in input order (-1 for padding). Counters: hits += k' - m,
 *      misses += m, evictions += #{u >= 0}, bytes += m * row_bytes (k' = non-padding entries).
 *
 * Three-tier variant ("Hybrid HiSparse" knowledge card, Timeline: one fused pass resolves resident, hot and
 * missing rows, the hot pages coming from ordinary KV blocks of the same memory pool). With a resident map, a
 * selected token that is not in the hot buffer but still held in the ordinary HBM KV pool (resident[t] = its row
 * there, >= 0) is served in place: it is neither a hit nor a miss, takes no slot, refreshes no stamp, and its
 * out_slot is -2 - resident[t]. It counts under hits (nothing is fetched). A hot-buffer hit takes precedence.
 *
 * The readings of points the paper leaves open (stamp = decode step number, ties by lowest slot, ascending-token
 * pairing, empties first, padding and rejection rules) are the ones listed in the design notes of this
 * repository. The code below follows the steps literally with library sorts (qsort); it is deliberately slow.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_ERR_RANGE 1
#define ORA_ERR_DUP 2

typedef struct {
  int32_t stamp;
  int32_t slot;
} ora_cand;

static int cmp_i32(const void *a, const void *b) {
  const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

static int cmp_cand(const void *a, const void *b) {
  const ora_cand *x = (const ora_cand *)a, *y = (const ora_cand *)b;
  if (x->stamp != y->stamp) return (x->stamp > y->stamp) - (x->stamp < y->stamp);
  return (x->slot > y->slot) - (x->slot < y->slot);
}

/*
 * One request-layer, one call. hot may be NULL (row bytes not tracked); host_rows may be NULL only if hot is.
 * counters: [hits, misses, evictions, bytes] accumulated. Returns 0, or an OR of ORA_ERR_* bits (row rejected),
 * -1 on allocation failure, -2 if k > slots.
 */
int ora_resolve_rl_tiered(int32_t step, int32_t ctx, int32_t slots, int32_t row_bytes, int32_t *tok2slot,
                          int32_t *slot_tok, int32_t *slot_stamp, uint8_t *hot, const uint8_t *host_rows,
                          const int32_t *sel, int32_t k, const int32_t *resident, int32_t *out_slots,
                          uint64_t *counters) {
  /* precondition: a selection never exceeds the cache (the library rejects k > slots before launching) */
  if (k > slots) return -2;
  /* 0. validation */
  int err = 0;
  int32_t *sorted = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
  if (!sorted) return -1;
  int32_t nvalid = 0;
  for (int32_t i = 0; i < k; ++i) {
    if (sel[i] >= ctx) err |= ORA_ERR_RANGE;
    if (sel[i] >= 0) sorted[nvalid++] = sel[i];
  }
  qsort(sorted, (size_t)nvalid, sizeof(int32_t), cmp_i32);
  for (int32_t i = 1; i < nvalid; ++i)
    if (sorted[i] == sorted[i - 1] && sorted[i] < ctx) err |= ORA_ERR_DUP;
  if (err) {
    if (out_slots)
      for (int32_t i = 0; i < k; ++i) out_slots[i] = -1;
    free(sorted);
    return err;
  }

  /* 1. hit test: stamp hits, remember the selected slots */
  uint8_t *in_sel = (uint8_t *)calloc((size_t)slots, 1);
  int32_t *miss = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
  ora_cand *cand = (ora_cand *)malloc(sizeof(ora_cand) * (size_t)slots);
  if (!in_sel || !miss || !cand) {
    free(sorted), free(in_sel), free(miss), free(cand);
    return -1;
  }
  int32_t m = 0, hits = 0, inplace = 0;
  for (int32_t i = 0; i < k; ++i) {
    const int32_t t = sel[i];
    if (t < 0) continue;
    const int32_t s = tok2slot[t];
    if (s >= 0) {
      slot_stamp[s] = step;
      in_sel[s] = 1;
      ++hits;
    } else if (resident && resident[t] >= 0) {
      ++inplace; /* served in place from the HBM-resident tier */
    } else {
      miss[m++] = t;
    }
  }

  /* 2. misses in ascending token order */
  qsort(miss, (size_t)m, sizeof(int32_t), cmp_i32);

  /* 3. candidates = slots not selected, ordered by (stamp, slot) */
  int32_t nc = 0;
  for (int32_t v = 0; v < slots; ++v)
    if (!in_sel[v]) {
      cand[nc].stamp = slot_stamp[v];
      cand[nc].slot = v;
      ++nc;
    }
  qsort(cand, (size_t)nc, sizeof(ora_cand), cmp_cand);

  /* 4. assignment (m <= nc because k <= slots and the selection has no duplicates) */
  int32_t evictions = 0;
  for (int32_t j = 0; j < m; ++j) {
    const int32_t t = miss[j], v = cand[j].slot, u = slot_tok[v];
    if (u >= 0) {
      tok2slot[u] = -1;
      ++evictions;
    }
    tok2slot[t] = v;
    slot_tok[v] = t;
    slot_stamp[v] = step;
    if (hot) memcpy(hot + (size_t)v * (size_t)row_bytes, host_rows + (size_t)t * (size_t)row_bytes, (size_t)row_bytes);
  }

  /* 5. outputs in input order, counters */
  if (out_slots)
    for (int32_t i = 0; i < k; ++i) out_slots[i] = sel[i] < 0 ? -1 : tok2slot[sel[i]];
  if (out_slots && resident)
    for (int32_t i = 0; i < k; ++i)
      if (sel[i] >= 0 && out_slots[i] < 0) out_slots[i] = -2 - resident[sel[i]];
  counters[0] += (uint64_t)inplace;
  counters[0] += (uint64_t)hits;
  counters[1] += (uint64_t)m;
  counters[2] += (uint64_t)evictions;
  counters[3] += (uint64_t)m * (uint64_t)row_bytes;

  free(sorted), free(in_sel), free(miss), free(cand);
  return 0;
}

int ora_resolve_rl(int32_t step, int32_t ctx, int32_t slots, int32_t row_bytes, int32_t *tok2slot,
                   int32_t *slot_tok, int32_t *slot_stamp, uint8_t *hot, const uint8_t *host_rows,
                   const int32_t *sel, int32_t k, int32_t *out_slots, uint64_t *counters) {
  return ora_resolve_rl_tiered(step, ctx, slots, row_bytes, tok2slot, slot_tok, slot_stamp, hot, host_rows, sel, k,
                               NULL, out_slots, counters);
}

/*
 * A batch of request-layers of one layer, laid out contiguously: tok2slot [nb][ctx], slot_tok/slot_stamp
 * [nb][slots], hot [nb][slots][row_bytes] (or NULL), host rows of request b at host + b*host_req_stride,
 * selections [nb][k], out_slots [nb][k] (or NULL). Returns the OR of all per-row error bits (or a negative code).
 */
int ora_resolve_batch_tiered(int32_t step, int32_t ctx, int32_t slots, int32_t row_bytes, int32_t nb,
                             int32_t *tok2slot, int32_t *slot_tok, int32_t *slot_stamp, uint8_t *hot,
                             const uint8_t *host, int64_t host_req_stride, const int32_t *sel, int32_t k,
                             const int32_t *resident, int32_t *out_slots, uint64_t *counters) {
  int err = 0;
  for (int32_t b = 0; b < nb; ++b) {
    int r = ora_resolve_rl_tiered(step, ctx, slots, row_bytes, tok2slot + (size_t)b * (size_t)ctx,
                                  slot_tok + (size_t)b * (size_t)slots, slot_stamp + (size_t)b * (size_t)slots,
                                  hot ? hot + (size_t)b * (size_t)slots * (size_t)row_bytes : NULL,
                                  host ? host + (size_t)b * (size_t)host_req_stride : NULL,
                                  sel + (size_t)b * (size_t)k, k, resident ? resident + (size_t)b * (size_t)ctx : NULL,
                                  out_slots ? out_slots + (size_t)b * (size_t)k : NULL, counters);
    if (r < 0) return r;
    err |= r;
  }
  return err;
}

int ora_resolve_batch(int32_t step, int32_t ctx, int32_t slots, int32_t row_bytes, int32_t nb, int32_t *tok2slot,
                      int32_t *slot_tok, int32_t *slot_stamp, uint8_t *hot, const uint8_t *host,
                      int64_t host_req_stride, const int32_t *sel, int32_t k, int32_t *out_slots,
                      uint64_t *counters) {
  return ora_resolve_batch_tiered(step, ctx, slots, row_bytes, nb, tok2slot, slot_tok, slot_stamp, hot, host,
                                  host_req_stride, sel, k, NULL, out_slots, counters);
}
