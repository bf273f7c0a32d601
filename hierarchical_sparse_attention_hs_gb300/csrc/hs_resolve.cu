// Fused per-layer selection resolution for a hierarchical KV cache, sm_103a.
//
// Method: "HiSparse: Scaling Sparse-Attention Decoding with Hierarchical KV Cache Management" (Abstract): a
// fused CUDA kernel resolves each layer's selections -- hit detection, LRU replacement and host-to-device
// fetches -- inside the decode CUDA graph; only the missing rows that hit the top-k are fetched ("HiSparse"
// knowledge card, Timeline). The policy details (stamps = decode step, oldest stamp first with ties to the
// lowest slot, misses paired with victims in ascending token order, empties first) are stated in hs.h.
//
// One launch resolves one layer for `batch` request-layers. A request-layer is served by a thread-block
// cluster of `C` CTAs (C = 1, 2, 4 or 8, chosen by the host from the batch so that enough SMs issue host-link
// loads). Every CTA of the cluster computes the full resolution redundantly from the same inputs, which is
// deterministic, so the CTAs agree without exchanging data; a cluster barrier separates the last read of the
// shared metadata from the first write, and the writes (metadata, out_slots, row copies) are partitioned
// between the CTAs. There is no spin-wait anywhere.
//
// Per CTA, in shared memory:
//   1. load the selection row, the slot stamps and slot tokens; clear the hit bitmap;
//   2. gather tok2slot for every selected token (random 4-byte reads); mark hit slots in the bitmap, which
//      also exposes a token selected twice among the hits;
//   3. stable LSD radix sort (8-bit digits, warp match + per-warp digit tables) of the miss positions by
//      token; the first pass filters the misses out of the selection (compaction fused with the sort);
//   4. stable LSD radix sort of the non-selected slots by stamp - min stamp; the first m are the victims in
//      (stamp, slot) order, because the sort is stable over slot order;
//   5. after the cluster barrier: hit stamps, miss assignment (unmap old token, map new, stamp), out_slots,
//      counters; then the row copies as 16-byte vector loads from mapped host memory (ld.global.cv, so a
//      host row is always fetched over the link, never served from a stale L2 line) straight into the hot
//      buffer, COPY_UNROLL independent loads in flight per thread.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/hs.h"

namespace {

constexpr int NT = 512;                 // threads per CTA
constexpr int NW = NT / 32;             // warps per CTA
constexpr int RADIX = 256;              // digit values per radix pass
constexpr int TBL_STRIDE = RADIX + 1;   // padded per-warp digit table row
constexpr int COPY_UNROLL = 8;          // 16-byte loads in flight per thread in the copy loop
constexpr int MAX_CLUSTER = 8;

struct ResolveArgs {
  const int32_t* topk;      // [batch][k]
  int32_t* out_slots;       // [batch][k] or nullptr (prefetch)
  int32_t* tok2slot;        // layer base, [max_batch][ctx]
  int32_t* slot_tok;        // layer base, [max_batch][slots]
  int32_t* slot_stamp;      // layer base, [max_batch][slots]
  unsigned long long* counters;  // layer's 4 counters
  const int32_t* step;
  int32_t* err;
  const uint8_t* src;       // row source of this layer, request 0
  int64_t src_req_stride;
  uint8_t* hot;             // layer base, [max_batch][slots][row_bytes]
  int32_t k, ctx, slots, row_bytes;
  int32_t cluster;          // CTAs per request-layer
};

// Contexts up to this many selection units rank their misses with a shared-memory bitmap (one bit per unit plus
// a 16-bit running count per 32 units); longer contexts use the radix sort.
constexpr int BITMAP_MAX_CTX = 1 << 18;

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
  size_t sel, slot, stamp, stok, hit, mpos, rank, cidx, mscr, tbl, red, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline bool use_bitmap(int ctx) { return ctx <= BITMAP_MAX_CTX; }

__host__ __device__ inline SmemLayout smem_layout(int k, int slots, int ctx) {
  SmemLayout L;
  size_t o = 0;
  L.sel = o;   o = align16(o + sizeof(int32_t) * k);
  L.slot = o;  o = align16(o + sizeof(int32_t) * k);
  L.stamp = o; o = align16(o + sizeof(int32_t) * slots);
  L.stok = o;  o = align16(o + sizeof(int32_t) * slots);
  L.hit = o;   o = align16(o + sizeof(uint32_t) * ((slots + 31) / 32));
  L.mpos = o;  o = align16(o + sizeof(uint16_t) * k);
  L.rank = o;  o = align16(o + sizeof(uint16_t) * k);
  L.cidx = o;  o = align16(o + sizeof(uint16_t) * 2 * slots);
  L.mscr = o;
  if (use_bitmap(ctx)) {
    const size_t words = ((size_t)ctx + 31) / 32;
    o = align16(o + sizeof(uint32_t) * words);
    o = align16(o + sizeof(uint16_t) * words);
  } else {
    o = align16(o + sizeof(uint16_t) * 2 * k);
  }
  L.tbl = o;   o = align16(o + sizeof(int32_t) * NW * TBL_STRIDE);
  L.red = o;   o = align16(o + sizeof(int32_t) * 4 * (NW + 1));
  L.total = o;
  return L;
}

// ------------------------------------------------------------------------------------------------------------
// Block-wide helpers (NT threads).
// ------------------------------------------------------------------------------------------------------------
__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int s = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) s += red[w];
  __syncthreads();
  return s;
}

__device__ __forceinline__ unsigned block_or(unsigned v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_or_sync(0xffffffffu, v);
  if (lane == 0) red[warp] = (int)v;
  __syncthreads();
  unsigned s = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) s |= (unsigned)red[w];
  __syncthreads();
  return s;
}

// min and max of non-negative ints in one pass (v < 0 means "no value").
__device__ __forceinline__ void block_minmax(int lo, int hi, int* red, int* out_lo, int* out_hi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  lo = (int)__reduce_min_sync(0xffffffffu, (unsigned)lo);  // unsigned: "no value" (INT_MAX) stays largest
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    red[warp] = lo;
    red[NW + 1 + warp] = hi;
  }
  __syncthreads();
  int a = 0x7fffffff, b = -1;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    a = min(a, red[w]);
    b = max(b, red[NW + 1 + w]);
  }
  __syncthreads();
  *out_lo = a;
  *out_hi = b;
}

// Exclusive prefix sum over the block; *total receives the sum of all values.
__device__ __forceinline__ int block_exclusive_scan(int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) red[lane] = w;
  }
  __syncthreads();
  const int before = warp ? red[warp - 1] : 0;
  *total = red[NW - 1];
  __syncthreads();
  return before + x - v;
}

// One stable counting-sort pass on the 8-bit digit at `shift`. Items come in order from `in` (or are the
// indices 0..n-1 when in == nullptr), items failing keep() are dropped, and the survivors are written to `out`
// grouped by digit, keeping their input order within a digit. Each warp owns a contiguous segment of the
// input and its own digit-count row, so ranks are exact and deterministic without atomics. Returns the number
// of survivors (the same on every thread).
template <class Key, class Keep>
__device__ int radix_pass(const uint16_t* __restrict__ in, int n, uint16_t* __restrict__ out, int shift, Key key,
                          Keep keep, int* __restrict__ tbl, int* __restrict__ red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (n + NW - 1) / NW;
  const int beg = min(n, warp * seg);
  const int end = min(n, beg + seg);
  int* wt = tbl + warp * TBL_STRIDE;
  for (int d = lane; d < RADIX; d += 32) wt[d] = 0;
  __syncwarp();
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    int item = 0;
    unsigned dig = RADIX;
    if (i < end) {
      item = in ? (int)in[i] : i;
      if (keep(item)) dig = ((unsigned)key(item) >> shift) & (RADIX - 1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, dig);
    if (dig < RADIX && lane == __ffs(peers) - 1) wt[dig] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // exclusive scan of the counts in (digit, warp) order
  constexpr int PER = RADIX * NW / NT;
  int cnt[PER];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = threadIdx.x * PER + e;
    cnt[e] = tbl[(idx % NW) * TBL_STRIDE + idx / NW];
    sum += cnt[e];
  }
  int total;
  int run = block_exclusive_scan(sum, red, &total);
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = threadIdx.x * PER + e;
    tbl[(idx % NW) * TBL_STRIDE + idx / NW] = run;
    run += cnt[e];
  }
  __syncthreads();
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    int item = 0;
    unsigned dig = RADIX;
    if (i < end) {
      item = in ? (int)in[i] : i;
      if (keep(item)) dig = ((unsigned)key(item) >> shift) & (RADIX - 1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, dig);
    if (dig < RADIX) out[wt[dig] + __popc(peers & ((1u << lane) - 1u))] = (uint16_t)item;
    __syncwarp();
    if (dig < RADIX && lane == __ffs(peers) - 1) wt[dig] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  return total;
}

// Full stable sort: pass 0 filters from the identity sequence 0..n-1 into buf[0]; further passes ping-pong.
// Returns a pointer to the buffer holding the result and its length in *count.
template <class Key, class Keep>
__device__ uint16_t* radix_sort(int n, int key_bits, uint16_t* buf0, uint16_t* buf1, Key key, Keep keep, int* tbl,
                                int* red, int* count) {
  int c = radix_pass(nullptr, n, buf0, 0, key, keep, tbl, red);
  uint16_t* cur = buf0;
  uint16_t* nxt = buf1;
  for (int shift = 8; shift < key_bits; shift += 8) {
    radix_pass(cur, c, nxt, shift, key, [](int) { return true; }, tbl, red);
    uint16_t* t = cur;
    cur = nxt;
    nxt = t;
  }
  *count = c;
  return cur;
}

// Order-preserving compaction of the indices i in [0, n) with pred(i) into out; returns the count (same on all
// threads). Each warp owns a contiguous segment; a ballot gives the in-warp offsets.
template <class Pred>
__device__ int block_compact(int n, uint16_t* __restrict__ out, Pred pred, int* __restrict__ red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (n + NW - 1) / NW;
  const int beg = min(n, warp * seg);
  const int end = min(n, beg + seg);
  int c = 0;
  for (int i = beg + lane; i < end; i += 32) c += pred(i) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) red[warp] = c;
  __syncthreads();
  int run = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int x = red[w];
    run += w < warp ? x : 0;
    total += x;
  }
  __syncthreads();
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const bool f = i < end && pred(i);
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (f) out[run + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)i;
    run += __popc(bal);
  }
  __syncthreads();
  return total;
}

// Rank of every miss among the misses by token, with a bitmap over the context: rank(t) = number of set bits
// below t = running count of the word holding t + popcount of its lower bits. Also flags a token set twice.
// mpos: miss positions (m of them); sel: selection row; rank_of_pos[pos] receives the rank.
__device__ unsigned bitmap_ranks(int m, int ctx, const uint16_t* __restrict__ mpos, const int32_t* __restrict__ sel,
                                 uint16_t* __restrict__ rank_of_pos, uint32_t* __restrict__ bits,
                                 uint16_t* __restrict__ prefix, int* __restrict__ red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwords = (ctx + 31) >> 5;
  unsigned bad = 0;
  for (int w = threadIdx.x; w < nwords; w += NT) bits[w] = 0u;
  __syncthreads();
  for (int q = threadIdx.x; q < m; q += NT) {
    const int t = sel[mpos[q]];
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bits[t >> 5], bit) & bit) bad |= HS_DEVERR_DUP;
  }
  __syncthreads();
  const int seg = (nwords + NW - 1) / NW;
  const int beg = min(nwords, warp * seg);
  const int end = min(nwords, beg + seg);
  int c = 0;
  for (int w = beg + lane; w < end; w += 32) c += __popc(bits[w]);
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) red[warp] = c;
  __syncthreads();
  int run = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) run += w < warp ? red[w] : 0;
  __syncthreads();
  for (int base = beg; base < end; base += 32) {
    const int w = base + lane;
    const int p = w < end ? __popc(bits[w]) : 0;
    int incl = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (w < end) prefix[w] = (uint16_t)(run + incl - p);
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncthreads();
  for (int q = threadIdx.x; q < m; q += NT) {
    const int pos = mpos[q];
    const int t = sel[pos];
    const int w = t >> 5;
    rank_of_pos[pos] = (uint16_t)(prefix[w] + __popc(bits[w] & ((1u << (t & 31)) - 1u)));
  }
  __syncthreads();
  return bad;
}

__device__ __forceinline__ int bits_of(unsigned x) { return x ? 32 - __clz(x) : 0; }

__device__ __forceinline__ uint4 load_row_chunk_host(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.cv.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 load_row_chunk_device(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

template <bool FROM_HOST>
__device__ __forceinline__ uint4 load_row_chunk(const uint8_t* p) {
  return FROM_HOST ? load_row_chunk_host(p) : load_row_chunk_device(p);
}

template <bool FROM_HOST, bool BITMAP>
__global__ void __launch_bounds__(NT, 1) hs_resolve_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const SmemLayout L = smem_layout(a.k, a.slots, a.ctx);
  int32_t* s_sel = reinterpret_cast<int32_t*>(smem + L.sel);
  int32_t* s_slot = reinterpret_cast<int32_t*>(smem + L.slot);
  int32_t* s_stamp = reinterpret_cast<int32_t*>(smem + L.stamp);
  int32_t* s_stok = reinterpret_cast<int32_t*>(smem + L.stok);
  uint32_t* s_hit = reinterpret_cast<uint32_t*>(smem + L.hit);
  uint16_t* s_mpos = reinterpret_cast<uint16_t*>(smem + L.mpos);
  uint16_t* s_rank = reinterpret_cast<uint16_t*>(smem + L.rank);
  uint16_t* s_cidx = reinterpret_cast<uint16_t*>(smem + L.cidx);
  uint8_t* s_mscr = smem + L.mscr;
  int* s_tbl = reinterpret_cast<int*>(smem + L.tbl);
  int* s_red = reinterpret_cast<int*>(smem + L.red);

  // Programmatic dependent launch: wait until the preceding kernel in the stream has completed and its writes
  // are visible, then let the next kernel start its launch while this one runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const int C = a.cluster;
  const int rank = blockIdx.x % C;
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int k = a.k, H = a.slots, ctx = a.ctx, R = a.row_bytes;
  const int32_t step = __ldcg(a.step);
  int32_t* t2s = a.tok2slot + (size_t)b * ctx;
  int32_t* s2t = a.slot_tok + (size_t)b * H;
  int32_t* stp = a.slot_stamp + (size_t)b * H;
  const int32_t* sel = a.topk + (size_t)b * k;
  int32_t* out = a.out_slots ? a.out_slots + (size_t)b * k : nullptr;
  const uint8_t* src = a.src + (size_t)b * (size_t)a.src_req_stride;
  uint8_t* hot = a.hot + (size_t)b * (size_t)H * (size_t)R;

  // 1. selection row, slot metadata, empty hit bitmap
  unsigned bad = 0;
  for (int i = tid; i < k; i += NT) {
    const int32_t t = __ldcg(sel + i);
    s_sel[i] = t;
    if (t >= ctx) bad |= HS_DEVERR_RANGE;
  }
  for (int v = tid; v < H; v += NT) {
    s_stamp[v] = __ldcg(stp + v);
    s_stok[v] = __ldcg(s2t + v);
  }
  for (int w = tid; w < (H + 31) / 32; w += NT) s_hit[w] = 0u;
  __syncthreads();

  // 2. hit test
  for (int i = tid; i < k; i += NT) {
    const int32_t t = s_sel[i];
    int32_t s = (t >= 0 && t < ctx) ? __ldcg(t2s + t) : -1;
    if (s >= H) {
      bad |= HS_DEVERR_STATE;
      s = -1;
    }
    s_slot[i] = s;
    if (s >= 0) {
      const uint32_t bit = 1u << (s & 31);
      if (atomicOr(&s_hit[s >> 5], bit) & bit) bad |= HS_DEVERR_DUP;
    }
  }
  __syncthreads();
  // Every read of the cluster-shared metadata by this CTA has completed.
  if (C > 1) cluster_arrive();

  // 3. misses in selection order
  auto is_miss = [&](int i) { return s_slot[i] < 0 && s_sel[i] >= 0 && s_sel[i] < ctx; };
  const int m = block_compact(k, s_mpos, is_miss, s_red);

  // 4. start this CTA's first wave of row loads now, so the host link is busy while the ranks and victims are
  //    being worked out; chunk c is 16-byte chunk (c % cpr) of the (c / cpr)-th miss in selection order
  const int cpr = R >> 4;
  const long long nchunk = (long long)m * cpr;
  const long long stride = (long long)C * NT;
  const long long c_first = (long long)rank * NT + tid;
  uint4 pre[COPY_UNROLL];
#pragma unroll
  for (int u = 0; u < COPY_UNROLL; ++u) {
    const long long c = c_first + u * stride;
    if (c < nchunk) {
      const int q = (int)(c / cpr);
      const int w = (int)(c - (long long)q * cpr);
      pre[u] = load_row_chunk<FROM_HOST>(src + (size_t)s_sel[s_mpos[q]] * (size_t)R + ((size_t)w << 4));
    }
  }

  // 5. rank of each miss among the misses by token
  if (BITMAP) {
    uint32_t* bits = reinterpret_cast<uint32_t*>(s_mscr);
    uint16_t* prefix = reinterpret_cast<uint16_t*>(s_mscr + align16(sizeof(uint32_t) * (size_t)((ctx + 31) >> 5)));
    bad |= bitmap_ranks(m, ctx, s_mpos, s_sel, s_rank, bits, prefix, s_red);
  } else {
    uint16_t* mbuf = reinterpret_cast<uint16_t*>(s_mscr);
    int m2 = 0;
    const uint16_t* midx = radix_sort(
        m, bits_of((unsigned)(ctx - 1)), mbuf, mbuf + k, [&](int q) { return s_sel[s_mpos[q]]; },
        [](int) { return true; }, s_tbl, s_red, &m2);
    for (int j = tid; j < m; j += NT) {
      const int pos = s_mpos[midx[j]];
      s_rank[pos] = (uint16_t)j;
      if (j && s_sel[pos] == s_sel[s_mpos[midx[j - 1]]]) bad |= HS_DEVERR_DUP;
    }
    __syncthreads();
  }

  // 6. victims: non-selected slots by (stamp, slot)
  int lo = 0x7fffffff, hi = -1;
  for (int v = tid; v < H; v += NT) {
    if (!(s_hit[v >> 5] & (1u << (v & 31)))) {
      lo = min(lo, s_stamp[v]);
      hi = max(hi, s_stamp[v]);
    }
  }
  int smin, smax;
  block_minmax(lo, hi, s_red, &smin, &smax);
  int ncand = 0;
  const int stamp_bits = smax >= smin ? bits_of((unsigned)(smax - smin)) : 0;
  const uint16_t* cidx = radix_sort(
      H, stamp_bits, s_cidx, s_cidx + H, [&](int v) { return s_stamp[v] - smin; },
      [&](int v) { return !(s_hit[v >> 5] & (1u << (v & 31))); }, s_tbl, s_red, &ncand);
  if (m > ncand) bad |= HS_DEVERR_STATE;
  bad = block_or(bad, s_red);

  if (C > 1) cluster_wait();  // no CTA of the cluster writes metadata before all have read it

  if (bad) {
    for (int i = rank * NT + tid; i < k; i += C * NT)
      if (out) out[i] = -1;
    if (rank == 0 && tid == 0) atomicOr(a.err, (int)bad);
    return;
  }

  // 7a. hits: stamp and emit
  for (int i = rank * NT + tid; i < k; i += C * NT) {
    const int32_t s = s_slot[i];
    if (s >= 0) stp[s] = step;
    if (out && (s >= 0 || s_sel[i] < 0)) out[i] = s;
  }
  // 7b. misses: the j-th smallest token takes the j-th victim
  int nevict = 0;
  for (int q = rank * NT + tid; q < m; q += C * NT) {
    const int pos = s_mpos[q];
    const int32_t t = s_sel[pos];
    const int32_t v = cidx[s_rank[pos]];
    const int32_t u = s_stok[v];
    if (u >= 0) {
      t2s[u] = -1;
      ++nevict;
    }
    t2s[t] = v;
    s2t[v] = t;
    stp[v] = step;
    if (out) out[pos] = v;
  }
  // 7c. the first wave of rows lands in its slots
#pragma unroll
  for (int u = 0; u < COPY_UNROLL; ++u) {
    const long long c = c_first + u * stride;
    if (c < nchunk) {
      const int q = (int)(c / cpr);
      const int w = (int)(c - (long long)q * cpr);
      const size_t v = cidx[s_rank[s_mpos[q]]];
      *reinterpret_cast<uint4*>(hot + v * (size_t)R + ((size_t)w << 4)) = pre[u];
    }
  }
  // 7d. the remaining rows, COPY_UNROLL loads in flight per thread
  for (long long c0 = c_first + stride * COPY_UNROLL; c0 < nchunk; c0 += stride * COPY_UNROLL) {
    uint4 v[COPY_UNROLL];
    uint8_t* dst[COPY_UNROLL];
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u) {
      const long long c = c0 + u * stride;
      dst[u] = nullptr;
      if (c < nchunk) {
        const int q = (int)(c / cpr);
        const int w = (int)(c - (long long)q * cpr);
        const int pos = s_mpos[q];
        v[u] = load_row_chunk<FROM_HOST>(src + (size_t)s_sel[pos] * (size_t)R + ((size_t)w << 4));
        dst[u] = hot + (size_t)cidx[s_rank[pos]] * (size_t)R + ((size_t)w << 4);
      }
    }
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u)
      if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = v[u];
  }
  nevict = block_sum(nevict, s_red);
  int nvalid = 0;
  for (int i = tid; i < k; i += NT) nvalid += s_sel[i] >= 0 ? 1 : 0;
  nvalid = block_sum(nvalid, s_red);
  if (tid == 0) {
    if (nevict) atomicAdd(a.counters + 2, (unsigned long long)nevict);
    if (rank == 0) {
      atomicAdd(a.counters + 0, (unsigned long long)(nvalid - m));
      atomicAdd(a.counters + 1, (unsigned long long)m);
      atomicAdd(a.counters + 3, (unsigned long long)m * (unsigned long long)R);
    }
  }
}

__global__ void hs_step_kernel(int32_t* step) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) *step += 1;
}

// Streaming read of n16 16-byte chunks from (mapped host or device) memory, COPY_UNROLL loads in flight per
// thread; the XOR of the data is written only if it matches an impossible value, so the loads stay live.
__global__ void hs_probe_read_kernel(const uint8_t* __restrict__ src, size_t n16, unsigned* __restrict__ sink) {
  const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t nth = (size_t)gridDim.x * blockDim.x;
  unsigned acc = 0;
  size_t i = tid;
  for (; i + (COPY_UNROLL - 1) * nth < n16; i += COPY_UNROLL * nth) {
    uint4 v[COPY_UNROLL];
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u) v[u] = load_row_chunk_host(src + ((i + u * nth) << 4));
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += nth) {
    const uint4 v = load_row_chunk_host(src + (i << 4));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) sink[0] = acc;
}

}  // namespace

// --------------------------------------------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------------------------------------------
struct hs_pool {
  hs_pool_desc d;
  hs_meta_layout lay;
  int device;
  int num_sms;
  bool noio;
  const uint8_t* src;  // device-visible row source
  int32_t* step;
  int32_t* err;
  unsigned long long* counters;
  int32_t* tok2slot;
  int32_t* slot_tok;
  int32_t* slot_stamp;
  size_t smem;
  int max_cluster;  // largest cluster size that fits on the device for this shared-memory size
};

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool geometry_ok(const hs_pool_desc* d) {
  if (!d) return false;
  if (d->layers < 1 || d->max_batch < 1 || d->ctx < 1 || d->slots < 1 || d->topk_max < 1) return false;
  if (d->topk_max > d->slots || d->slots > 65535) return false;
  if (d->row_bytes <= 0 || (d->row_bytes & 15)) return false;
  if (d->host_layer_stride < 0 || (d->host_layer_stride & 15)) return false;
  if (d->host_req_stride < 0 || (d->host_req_stride & 15)) return false;
  return true;
}

bool layout_of(const hs_pool_desc* d, hs_meta_layout* L) {
  if (!geometry_ok(d)) return false;
  const size_t rl = (size_t)d->layers * (size_t)d->max_batch;
  size_t o = 0;
  L->step = o;
  L->error = o + 4;
  o = 256;
  L->counters = o;
  o = align256(o + sizeof(uint64_t) * 4 * (size_t)d->layers);
  L->tok2slot = o;
  o = align256(o + sizeof(int32_t) * rl * (size_t)d->ctx);
  L->slot_tok = o;
  o = align256(o + sizeof(int32_t) * rl * (size_t)d->slots);
  L->slot_stamp = o;
  o = align256(o + sizeof(int32_t) * rl * (size_t)d->slots);
  L->total = o;
  return true;
}

// Device-visible address of page-locked (cudaHostAlloc / cudaHostRegister) host memory, or nullptr. Plain
// pageable memory is refused even where the GPU could reach it through the CPU's page tables: the host tier
// must stay resident while kernels read it.
const void* mapped_host_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost) return nullptr;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return d;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

int init_meta(hs_pool* p, cudaStream_t s) {
  uint8_t* base = static_cast<uint8_t*>(p->d.meta);
  const size_t rl = (size_t)p->d.layers * (size_t)p->d.max_batch;
  if (cudaMemsetAsync(base, 0, p->lay.tok2slot, s) != cudaSuccess) return HS_ERR_CUDA;  // header + counters
  if (cudaMemsetAsync(base + p->lay.tok2slot, 0xff, sizeof(int32_t) * rl * (size_t)p->d.ctx, s) != cudaSuccess)
    return HS_ERR_CUDA;
  if (cudaMemsetAsync(base + p->lay.slot_tok, 0xff, sizeof(int32_t) * rl * (size_t)p->d.slots, s) != cudaSuccess)
    return HS_ERR_CUDA;
  if (cudaMemsetAsync(base + p->lay.slot_stamp, 0, sizeof(int32_t) * rl * (size_t)p->d.slots, s) != cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

int pick_cluster(const hs_pool* p, int batch) {
  // Enough CTAs to keep the host link (or HBM, in no-IO mode) busy; the link saturates with a few dozen SMs.
  const int target = p->noio ? p->num_sms : 64;
  int c = 1;
  while (c < p->max_cluster && batch * c < target) c <<= 1;
  return c;
}

int launch_resolve(hs_pool* p, int32_t layer, int32_t batch, const int32_t* topk, int32_t k, int32_t* out,
                   cudaStream_t s) {
  if (!p || layer < 0 || layer >= p->d.layers || batch < 0 || batch > p->d.max_batch || k < 0 ||
      k > p->d.topk_max)
    return HS_ERR_INVALID_ARG;
  if (batch == 0 || k == 0) return HS_OK;
  if (!topk) return HS_ERR_INVALID_ARG;
  const size_t rl0 = (size_t)layer * (size_t)p->d.max_batch;
  ResolveArgs a;
  a.topk = topk;
  a.out_slots = out;
  a.tok2slot = p->tok2slot + rl0 * (size_t)p->d.ctx;
  a.slot_tok = p->slot_tok + rl0 * (size_t)p->d.slots;
  a.slot_stamp = p->slot_stamp + rl0 * (size_t)p->d.slots;
  a.counters = p->counters + 4 * (size_t)layer;
  a.step = p->step;
  a.err = p->err;
  a.src = p->src + (size_t)layer * (size_t)p->d.host_layer_stride;
  a.src_req_stride = p->d.host_req_stride ? p->d.host_req_stride : (int64_t)p->d.ctx * p->d.row_bytes;
  a.hot = static_cast<uint8_t*>(p->d.hot_buf) + rl0 * (size_t)p->d.slots * (size_t)p->d.row_bytes;
  a.k = k;
  a.ctx = p->d.ctx;
  a.slots = p->d.slots;
  a.row_bytes = p->d.row_bytes;
  a.cluster = pick_cluster(p, batch);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(batch * a.cluster), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem_layout(k, p->d.slots, p->d.ctx).total;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (a.cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)a.cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  const bool bm = use_bitmap(p->d.ctx);
  cudaError_t e;
  if (p->noio)
    e = bm ? cudaLaunchKernelEx(&cfg, hs_resolve_kernel<false, true>, a)
           : cudaLaunchKernelEx(&cfg, hs_resolve_kernel<false, false>, a);
  else
    e = bm ? cudaLaunchKernelEx(&cfg, hs_resolve_kernel<true, true>, a)
           : cudaLaunchKernelEx(&cfg, hs_resolve_kernel<true, false>, a);
  return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t hs_meta_bytes(const hs_pool_desc* desc) {
  hs_meta_layout L;
  return layout_of(desc, &L) ? L.total : 0;
}

int hs_get_meta_layout(const hs_pool_desc* desc, hs_meta_layout* out) {
  if (!out || !layout_of(desc, out)) return HS_ERR_INVALID_ARG;
  return HS_OK;
}

int hs_pool_create(const hs_pool_desc* desc, hs_stream_t stream, hs_pool** out) {
  if (!out) return HS_ERR_INVALID_ARG;
  *out = nullptr;
  hs_meta_layout lay;
  if (!layout_of(desc, &lay)) return HS_ERR_INVALID_ARG;
  if (!desc->hot_buf || !desc->meta || (reinterpret_cast<uintptr_t>(desc->hot_buf) & 15) ||
      (reinterpret_cast<uintptr_t>(desc->meta) & 255))
    return HS_ERR_INVALID_ARG;
  if (!is_device_ptr(desc->hot_buf) || !is_device_ptr(desc->meta)) return HS_ERR_INVALID_ARG;
  const uint8_t* src = nullptr;
  if (desc->noio_src) {
    if ((reinterpret_cast<uintptr_t>(desc->noio_src) & 15) || !is_device_ptr(desc->noio_src))
      return HS_ERR_INVALID_ARG;
    src = static_cast<const uint8_t*>(desc->noio_src);
  } else {
    if (!desc->host_pool || (reinterpret_cast<uintptr_t>(desc->host_pool) & 15)) return HS_ERR_INVALID_ARG;
    const void* dptr = mapped_host_ptr(desc->host_pool);
    if (!dptr) return HS_ERR_NOT_MAPPED;
    src = static_cast<const uint8_t*>(dptr);
  }
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return HS_ERR_CUDA;
  const size_t smem = smem_layout(desc->topk_max, desc->slots, desc->ctx).total;
  if (smem > (size_t)optin) return HS_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(hs_resolve_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
          cudaSuccess ||
      cudaFuncSetAttribute(hs_resolve_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
          cudaSuccess ||
      cudaFuncSetAttribute(hs_resolve_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
          cudaSuccess ||
      cudaFuncSetAttribute(hs_resolve_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
          cudaSuccess)
    return HS_ERR_CUDA;

  hs_pool* p = new (std::nothrow) hs_pool;
  if (!p) return HS_ERR_NO_MEMORY;
  p->d = *desc;
  p->lay = lay;
  p->device = dev;
  p->num_sms = sms;
  p->noio = desc->noio_src != nullptr;
  p->src = src;
  uint8_t* base = static_cast<uint8_t*>(desc->meta);
  p->step = reinterpret_cast<int32_t*>(base + lay.step);
  p->err = reinterpret_cast<int32_t*>(base + lay.error);
  p->counters = reinterpret_cast<unsigned long long*>(base + lay.counters);
  p->tok2slot = reinterpret_cast<int32_t*>(base + lay.tok2slot);
  p->slot_tok = reinterpret_cast<int32_t*>(base + lay.slot_tok);
  p->slot_stamp = reinterpret_cast<int32_t*>(base + lay.slot_stamp);
  p->smem = smem;
  // largest power-of-two cluster whose CTAs fit on the device at this shared-memory size
  p->max_cluster = 1;
  for (int c = 2; c <= MAX_CLUSTER; c <<= 1) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)c, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)c;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, hs_resolve_kernel<true, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      break;
    }
    if (n < 1) break;
    p->max_cluster = c;
  }
  const int rc = init_meta(p, reinterpret_cast<cudaStream_t>(stream));
  if (rc != HS_OK) {
    delete p;
    return rc;
  }
  *out = p;
  return HS_OK;
}

int hs_pool_reset(hs_pool* pool, hs_stream_t stream) {
  if (!pool) return HS_ERR_INVALID_ARG;
  return init_meta(pool, reinterpret_cast<cudaStream_t>(stream));
}

int hs_step_begin(hs_pool* pool, hs_stream_t stream) {
  if (!pool) return HS_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hs_step_kernel, pool->step) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_resolve(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* topk_idx, int32_t k,
               int32_t* out_slots, hs_stream_t stream) {
  if (batch > 0 && k > 0 && !out_slots) return HS_ERR_INVALID_ARG;
  return launch_resolve(pool, layer, batch, topk_idx, k, out_slots, reinterpret_cast<cudaStream_t>(stream));
}

int hs_prefetch(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* topk_idx, int32_t k,
                hs_stream_t stream) {
  return launch_resolve(pool, layer, batch, topk_idx, k, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int hs_get_error(hs_pool* pool, int32_t* out, int32_t clear) {
  if (!pool || !out) return HS_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemcpy(out, pool->err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return HS_ERR_CUDA;
  if (clear && cudaMemset(pool->err, 0, sizeof(int32_t)) != cudaSuccess) return HS_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  return HS_OK;
}

int hs_get_counters(hs_pool* pool, int32_t layer, uint64_t out[4]) {
  if (!pool || !out || layer < 0 || layer >= pool->d.layers) return HS_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemcpy(out, pool->counters + 4 * (size_t)layer, 4 * sizeof(uint64_t), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

int hs_pool_destroy(hs_pool* pool) {
  if (!pool) return HS_ERR_INVALID_ARG;
  delete pool;
  return HS_OK;
}

int hs_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return HS_ERR_INVALID_ARG;
  *out = nullptr;
  if (cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    cudaGetLastError();
    *out = nullptr;
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

int hs_host_free(void* ptr) {
  if (!ptr) return HS_ERR_INVALID_ARG;
  return cudaFreeHost(ptr) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_probe_link(const void* host, void* dev, size_t bytes, int32_t iters, hs_stream_t stream,
                  double* zero_copy_gbs, double* memcpy_gbs) {
  if (!host || !dev || bytes < 16 || (bytes & 15) || iters < 1 || !zero_copy_gbs || !memcpy_gbs ||
      (reinterpret_cast<uintptr_t>(host) & 15))
    return HS_ERR_INVALID_ARG;
  const void* dhost = mapped_host_ptr(host);
  if (!dhost) return HS_ERR_NOT_MAPPED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev_id = 0, sms = 0;
  if (cudaGetDevice(&dev_id) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_id) != cudaSuccess)
    return HS_ERR_CUDA;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return HS_ERR_CUDA;
  }
  int rc = HS_OK;
  float best_zc = 1e30f, best_cp = 1e30f, ms = 0.f;
  for (int r = 0; r <= iters && rc == HS_OK; ++r) {  // round 0 warms up
    if (cudaEventRecord(e0, s) != cudaSuccess) rc = HS_ERR_CUDA;
    hs_probe_read_kernel<<<2 * sms, 512, 0, s>>>(static_cast<const uint8_t*>(dhost), bytes >> 4,
                                                  static_cast<unsigned*>(dev));
    if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e1, s) != cudaSuccess ||
        cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      rc = HS_ERR_CUDA;
    if (r && ms < best_zc) best_zc = ms;
    if (rc != HS_OK) break;
    if (cudaEventRecord(e0, s) != cudaSuccess ||
        cudaMemcpyAsync(dev, host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      rc = HS_ERR_CUDA;
    if (r && ms < best_cp) best_cp = ms;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != HS_OK) return rc;
  *zero_copy_gbs = (double)bytes / (best_zc * 1e6);
  *memcpy_gbs = (double)bytes / (best_cp * 1e6);
  return HS_OK;
}

const char* hs_error_string(int code) {
  switch (code) {
    case HS_OK: return "ok";
    case HS_ERR_INVALID_ARG: return "invalid argument";
    case HS_ERR_CUDA: return "CUDA runtime error";
    case HS_ERR_NOT_MAPPED: return "host pool is not page-locked device-mapped memory";
    case HS_ERR_NO_MEMORY: return "out of host memory";
    case HS_ERR_UNSUPPORTED: return "geometry needs more shared memory than the device offers";
    default: return "unknown error";
  }
}

}  // extern "C"
