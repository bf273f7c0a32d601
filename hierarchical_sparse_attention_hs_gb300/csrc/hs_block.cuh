// Block- and warp-group-level building blocks of the resolve kernel (sm_103a): reductions, scans, ordered
// compaction, and a stable 8-bit counting-sort pass. A "group" is a contiguous range of warps of the CTA that
// synchronises on its own named barrier, so two groups can run different phases at the same time.
#pragma once

#include <cstdint>

namespace hs {

constexpr int NT = 512;               // threads per CTA
constexpr int NW = NT / 32;           // warps per CTA
constexpr int RADIX = 256;            // digit values per counting-sort pass
constexpr int TBL_STRIDE = RADIX + 1; // padded digit-count row per warp
constexpr int RED_INTS = 4 * (NW + 1);

struct Group {
  int w0;   // first warp
  int nw;   // warps
  int bar;  // named barrier id (0 = the whole CTA)
  __device__ __forceinline__ int warp() const { return (int)(threadIdx.x >> 5) - w0; }
  __device__ __forceinline__ int tid() const { return (int)threadIdx.x - w0 * 32; }
  __device__ __forceinline__ int size() const { return nw * 32; }
  __device__ __forceinline__ void sync() const {
    if (bar == 0)
      __syncthreads();
    else
      asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nw * 32) : "memory");
  }
};

__device__ __forceinline__ unsigned lanemask_lt() { return (1u << (threadIdx.x & 31)) - 1u; }

// Sum over the group; red: RED_INTS ints owned by the group.
__device__ __forceinline__ int group_sum(const Group& g, int v, int* red) {
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) red[g.warp()] = v;
  g.sync();
  int s = 0;
  for (int w = 0; w < g.nw; ++w) s += red[w];
  g.sync();
  return s;
}

__device__ __forceinline__ unsigned group_or(const Group& g, unsigned v, int* red) {
  v = __reduce_or_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) red[g.warp()] = (int)v;
  g.sync();
  unsigned s = 0;
  for (int w = 0; w < g.nw; ++w) s |= (unsigned)red[w];
  g.sync();
  return s;
}

// Exclusive prefix sum over the group in thread order; *total = sum of all values.
__device__ __forceinline__ int group_exclusive_scan(const Group& g, int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = g.warp();
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  g.sync();
  if (warp == 0) {
    int w = lane < g.nw ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < g.nw) red[lane] = w;
  }
  g.sync();
  const int before = warp ? red[warp - 1] : 0;
  *total = red[g.nw - 1];
  g.sync();
  return before + x - v;
}

// Order-preserving compaction of the indices i in [0, n) with pred(i) into out; returns the count. Each warp
// owns a contiguous segment; a ballot gives the offsets inside a warp.
template <class Pred>
__device__ int group_compact(const Group& g, int n, uint16_t* __restrict__ out, Pred pred, int* __restrict__ red) {
  const int lane = threadIdx.x & 31, warp = g.warp();
  const int seg = (n + g.nw - 1) / g.nw;
  const int beg = min(n, warp * seg);
  const int end = min(n, beg + seg);
  int c = 0;
  for (int i = beg + lane; i < end; i += 32) c += pred(i) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) red[warp] = c;
  g.sync();
  int run = 0, total = 0;
  for (int w = 0; w < g.nw; ++w) {
    const int x = red[w];
    run += w < warp ? x : 0;
    total += x;
  }
  g.sync();
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const bool f = i < end && pred(i);
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (f) out[run + __popc(bal & lanemask_lt())] = (uint16_t)i;
    run += __popc(bal);
  }
  g.sync();
  return total;
}

// Lanes of the warp whose digit equals this lane's, from one ballot per significant digit bit (dig < 2^nbits)
// plus one for `valid`; invalid lanes get an empty mask.
__device__ __forceinline__ unsigned digit_peers(unsigned dig, bool valid, int nbits) {
  unsigned peers = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool on = (dig >> b) & 1u;
    const unsigned m = __ballot_sync(0xffffffffu, on);
    peers &= on ? m : ~m;
  }
  return valid ? peers : 0u;
}

// One stable counting-sort pass on the digit (key >> shift) & (2^nbits - 1), nbits <= 8. Items come in order
// from `in` (or are 0..n-1 when in == nullptr); items failing keep() are dropped; survivors go to `out` grouped
// by digit, in input order within a digit. Each warp owns a contiguous input segment and a digit-count row of
// tbl (rows of the group's warps): counts by shared atomics (order-free), ranks inside a warp from ballots, so
// the order is exact and deterministic. Returns the survivor count.
//
// With limit >= 0, only the first `limit` output positions are needed: items whose digit lies above the digit
// holding position limit - 1 are not written, and a chunk of 32 items with none below it is skipped after one
// ballot. (Only meaningful for the last pass of a sort.)
template <class Key, class Keep>
__device__ int radix_pass(const Group& g, const uint16_t* __restrict__ in, int n, uint16_t* __restrict__ out,
                          int shift, int nbits, Key key, Keep keep, int* __restrict__ tbl, int* __restrict__ red,
                          int limit = -1) {
  const int lane = threadIdx.x & 31, warp = g.warp();
  const int seg = (n + g.nw - 1) / g.nw;
  const int beg = min(n, warp * seg);
  const int end = min(n, beg + seg);
  const unsigned dmask = (1u << nbits) - 1u;
  int* wt = tbl + (g.w0 + warp) * TBL_STRIDE;
  for (int d = lane; d < RADIX; d += 32) wt[d] = 0;
  __syncwarp();
  for (int i = beg + lane; i < end; i += 32) {
    const int item = in ? (int)in[i] : i;
    if (keep(item)) atomicAdd(&wt[((unsigned)key(item) >> shift) & dmask], 1);
  }
  g.sync();
  // exclusive scan of the counts in (digit, warp) order: RADIX * nw entries, 8 per thread
  constexpr int PER = RADIX / 32;
  const int* rows = tbl + g.w0 * TBL_STRIDE;
  int cnt[PER];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = g.tid() * PER + e;
    cnt[e] = rows[(idx % g.nw) * TBL_STRIDE + idx / g.nw];
    sum += cnt[e];
  }
  int total;
  int run = group_exclusive_scan(g, sum, red, &total);
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = g.tid() * PER + e;
    tbl[(g.w0 + idx % g.nw) * TBL_STRIDE + idx / g.nw] = run;
    run += cnt[e];
  }
  g.sync();
  // highest digit still needed: the one whose range of output positions holds position limit - 1
  unsigned top = dmask;
  if (limit >= 0) {
    if (limit == 0) {
      g.sync();
      return total;
    }
    const int* first = tbl + g.w0 * TBL_STRIDE;  // first warp's row: exclusive start of each digit
    int lo = 0, hi = (int)dmask;
    while (lo < hi) {  // largest d with start(d) <= limit - 1
      const int mid = (lo + hi + 1) >> 1;
      if (first[mid] <= limit - 1)
        lo = mid;
      else
        hi = mid - 1;
    }
    top = (unsigned)lo;
  }
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    int item = 0;
    unsigned dig = 0;
    bool valid = false;
    if (i < end) {
      item = in ? (int)in[i] : i;
      valid = keep(item);
      if (valid) dig = ((unsigned)key(item) >> shift) & dmask;
    }
    valid = valid && dig <= top;
    if (limit >= 0 && !__ballot_sync(0xffffffffu, valid)) continue;
    const unsigned peers = digit_peers(dig, valid, nbits);
    if (valid) out[wt[dig] + __popc(peers & lanemask_lt())] = (uint16_t)item;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wt[dig] += __popc(peers);
    __syncwarp();
  }
  g.sync();
  return total;
}

// Stable LSD sort on the low key_bits bits: pass 0 filters the identity sequence 0..n-1 into buf0, later passes
// ping-pong. Returns the buffer holding the result; *count = the number of items kept (with a limit, only the
// first `limit` positions of the result are guaranteed).
template <class Key, class Keep>
__device__ uint16_t* radix_sort(const Group& g, int n, int key_bits, uint16_t* buf0, uint16_t* buf1, Key key,
                                Keep keep, int* tbl, int* red, int* count, int limit = -1) {
  // a limit only applies to a single-pass sort (the pass that fixes the final order)
  int c = radix_pass(g, nullptr, n, buf0, 0, min(8, max(key_bits, 0)), key, keep, tbl, red,
                     key_bits <= 8 ? limit : -1);
  uint16_t* cur = buf0;
  uint16_t* nxt = buf1;
  for (int shift = 8; shift < key_bits; shift += 8) {
    radix_pass(g, cur, c, nxt, shift, min(8, key_bits - shift), key, [](int) { return true; }, tbl, red);
    uint16_t* t = cur;
    cur = nxt;
    nxt = t;
  }
  *count = c;
  return cur;
}

__device__ __forceinline__ int bits_of(unsigned x) { return x ? 32 - __clz(x) : 0; }

}  // namespace hs
