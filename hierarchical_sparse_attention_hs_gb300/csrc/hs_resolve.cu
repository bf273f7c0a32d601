// Fused per-layer selection resolution for a hierarchical KV cache, sm_103a.
//
// Method: "HiSparse: Scaling Sparse-Attention Decoding with Hierarchical KV Cache Management" (Abstract): for every
// layer, one kernel inside the decode step's CUDA graph looks the layer's selections up in a fixed-size GPU cache,
// replaces least recently used entries and fetches the missing rows from host memory; only missing rows that the
// top-k selects are brought over ("HiSparse" knowledge card, Timeline). The policy (stamps = decode step, oldest
// stamp first with ties to the lowest slot, misses paired with victims in ascending token order, empties first) is
// stated in hs.h.
//
// One launch resolves one layer for `batch` request-layers. A request-layer is served by a thread-block cluster of
// C CTAs (C = 1, 2, 4 or 8, chosen by the host so that enough SMs issue host-link loads while the grid stays within
// one wave). Every CTA reads the request-layer's selection, slot stamps and slot tokens and finds the hits and the
// misses itself; the victim choice is split between the CTAs and its pieces are exchanged through distributed
// shared memory (asynchronous remote stores counted by mbarrier transaction bytes); a cluster barrier separates
// the last read of the shared metadata from the first write; metadata writes and row copies are split by CTA.
// Every wait is bounded; bad input never traps (it sets the sticky error word).
//
// Per CTA (512 threads), in shared memory:
//   1. the slot stamps and slot tokens start for shared memory as asynchronous copies while each warp loads its
//      run of the selection row; the bitmaps and bucket counts are cleared and the exchange barriers set up;
//   2. each warp gathers tok2slot for its run of selection entries (random 4-byte reads, several in flight per
//      thread); a hit sets its slot's bit in the hit bitmap, a repeated slot or token is an error;
//   3. the misses in selection order, by ballots over the same runs (identical in every CTA of the cluster);
//   4. two warp groups at once, each on its own named barrier:
//      A (warps 0-7): at once the first wave of row loads from host memory into registers -- the link is busy
//         while the resolution goes on -- then the rank of every miss among the misses by token: a counting sort
//         of the miss tokens on their top bits (at most 2048 buckets), then the few smaller tokens in the bucket;
//      B (warps 8-15): the victims. CTA r of the cluster takes the r-th range of slots; one pass over it gives the
//         candidates' stamp range and, from ballot bit planes, how many candidates have each stamp modulo 32. The
//         rows of all CTAs are exchanged; when the candidates span at most 32 stamps these are exact per-stamp
//         counts, and the bin holding position m - 1 splits the bins taken whole from the one taken in slot
//         order. Each CTA scatters its range's victims, in (stamp, slot) order, into every CTA's victim list.
//         Wider stamp spans sort all candidates instead (stable LSD radix sort, in every CTA);
//   5. group A, after the cluster barrier, per owned selection entry (runs of 32 entries, round-robin over the
//      cluster): a hit is stamped; a miss of rank j takes victim j (the old token is unmapped, the new one mapped,
//      the slot stamped); out_slots in input order;
//   6. rows: the row chunks are split between the cluster's CTAs in interleaved runs of blocks of
//      32 x COPY_UNROLL chunks (a run covers a whole row when rows span several blocks); group B starts on this
//      CTA's blocks past the first wave at once (no other CTA reads the hot buffer, so this needs no barrier),
//      group A lands its first wave in the victims' slots after step 5 and joins; warps take blocks from a shared
//      counter. Loads are 16-byte ld.global.cv (a host row always comes over the link, never from a stale L2
//      line), straight into the hot buffer.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/hs.h"
#include "hs_block.cuh"
#include "hs_pool.hpp"

namespace {

using hs::bits_of;
using hs::Group;
using hs::NT;
using hs::NW;
using hs::RED_INTS;
using hs::TBL_STRIDE;

constexpr int COPY_UNROLL = 8;  // 16-byte loads in flight per thread in the copy loops
constexpr int MAX_CLUSTER = HS_MAX_CLUSTER;
constexpr int GA_WARPS = NW / 2;                 // group A: miss ranks and the first wave of row loads
constexpr int GA_THREADS = GA_WARPS * 32;
constexpr int BITMAP_MAX_CTX = 1 << 18;          // longer contexts rank misses with the radix sort
constexpr int MISC_BAD = 0, MISC_NCAND = 1, MISC_NEXT = 2, MISC_NINP = 3, MISC_XFAIL = 4, MISC_INTS = 5;
constexpr int NBUCKET = 2048;  // miss ranking: tokens are counted into at most this many buckets of 2^shift
constexpr int XROW = 36;       // victim choice: one warp's row = 32 stamp counts + (min, max, count, 0) stamps
constexpr int XROWS = MAX_CLUSTER * (NW - GA_WARPS);  // rows of the exchange table: every warp of group B
constexpr unsigned XWAIT_LIMIT = 1u << 22;  // polls of an exchange barrier before the call is given up

struct ResolveArgs {
  const int32_t* topk;           // [batch][k]
  int32_t* out_slots;            // [batch][k] or nullptr (prefetch)
  int32_t* tok2slot;             // layer base, [max_batch][ctx]
  int32_t* slot_tok;             // layer base, [max_batch][slots]
  int32_t* slot_stamp;           // layer base, [max_batch][slots]
  unsigned long long* counters;  // layer's 4 counters
  const int32_t* step;
  int32_t* err;
  // Fused step begin: this launch resolves at step + begin; the last of its CTAs to finish (counted in *done, which
  // it leaves at 0) stores the advanced step for the launches after it. 0 for an ordinary call.
  int32_t begin;
  int32_t* done;
  const uint8_t* src;            // row source of this layer, request 0
  int64_t src_req_stride;
  uint8_t* hot;                  // layer base, [max_batch][slots][row_bytes]
  int32_t k, ctx, slots, row_bytes;
  int32_t cluster;               // CTAs per request-layer
  // Layers resolved by this launch: layer 0 of the args and the nlayers - 1 after it, whose caches hold the same
  // metadata (they are always resolved together with one shared selection). Strides between layers.
  // Three-tier variant: row of each token still held in the ordinary HBM KV pool (>= 0) or -1, for request b at
  // resident + b * resident_stride; nullptr when there is no such tier.
  const int32_t* resident;
  int64_t resident_stride;
  int32_t nlayers;
  int32_t groups;                // layer groups: cluster (b, g) handles request b for the g-th run of layers
  const int32_t* req_ids;        // [batch] pool request of each batch row, or nullptr (row b is request b)
  int32_t max_batch;             // pool requests (valid request ids are 0 .. max_batch-1)
  int64_t meta_layer_ctx;        // int32 elements between layers in tok2slot
  int64_t meta_layer_slots;      // int32 elements between layers in slot_tok / slot_stamp
  int64_t src_layer_bytes;       // bytes between layers in the row source
  int64_t hot_layer_bytes;       // bytes between layers in the hot buffer
};

__host__ __device__ inline bool use_bitmap(int ctx) { return ctx <= BITMAP_MAX_CTX; }
__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Shared-memory carve-up, identical on host and device.
struct SmemLayout {
  size_t sel, slot, stamp, stok, hit, mpos, cidx, mscr, rank, bcnt, blist, vic, xrow, bar, tbl, red, wstat, misc,
      total;
};

__host__ __device__ inline SmemLayout smem_layout(int k, int slots, int ctx) {
  SmemLayout L;
  size_t o = 0;
  L.sel = o;   o = align16(o + sizeof(int32_t) * k);
  L.slot = o;  o = align16(o + sizeof(int32_t) * k);
  L.stamp = o; o = align16(o + sizeof(int32_t) * slots);
  L.stok = o;  o = align16(o + sizeof(int32_t) * slots);
  L.hit = o;   o = align16(o + sizeof(uint32_t) * ((slots + 31) / 32));
  L.mpos = o;  o = align16(o + sizeof(uint16_t) * k);
  L.cidx = o;  o = align16(o + sizeof(uint16_t) * 2 * slots);
  if (use_bitmap(ctx))
    L.mscr = o, o = align16(o + sizeof(uint32_t) * (((size_t)ctx + 31) / 32));  // token bitmap
  else
    L.mscr = o, o = align16(o + sizeof(uint16_t) * 2 * k);  // radix ping-pong (repeated in-place tokens)
  L.rank = o;  o = align16(o + sizeof(uint16_t) * k);         // rank of the miss at each selection entry
  L.bcnt = o;  o = align16(o + sizeof(int32_t) * NBUCKET);    // misses per token bucket, then bucket bounds
  L.blist = o; o = align16(o + sizeof(int32_t) * k);          // miss tokens grouped by bucket
  L.vic = o;   o = align16(o + sizeof(int32_t) * k);          // victim j, the slot of the miss of rank j
  L.xrow = o;  o = align16(o + sizeof(int32_t) * XROWS * XROW);
  L.bar = o;   o = align16(o + sizeof(uint64_t) * 2);          // exchange barriers: rows, victims
  L.tbl = o;   o = align16(o + sizeof(int32_t) * NW * TBL_STRIDE);
  L.red = o;   o = align16(o + sizeof(int32_t) * 2 * RED_INTS);
  L.wstat = o; o = align16(o + sizeof(int32_t) * 4 * NW);
  L.misc = o;  o = align16(o + sizeof(int32_t) * MISC_INTS);
  L.total = o;
  return L;
}

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

template <bool FROM_HOST>
__device__ __forceinline__ uint4 load_row_chunk(const uint8_t* p) {
  return FROM_HOST ? load_row_chunk_host(p) : load_row_chunk_device(p);
}

// Loads of the caller's index arrays (selections, resident maps, slot lists): `.cv` fetches afresh, so a stale
// L2 copy of a host-memory line is never used and these arrays may live in device memory or in mapped
// page-locked host memory, read over the host link without a separate copy.
__device__ __forceinline__ int32_t ld_fresh(const int32_t* p) {
  int32_t v;
  asm("ld.global.cv.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Asynchronous global-to-shared copies (completion waited for by the issuing thread, then a block barrier).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Every warp executes these as a whole (the .aligned forms). The arrive carries no release: it signals that
// this CTA's reads of the shared metadata have returned their values (loads consumed, copies waited for), which
// no later write of another CTA can change; there is nothing of this CTA's to publish at that point.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Exchanges between the CTAs of a cluster through distributed shared memory: asynchronous remote stores whose
// bytes complete the transaction count of the receiver's mbarrier, which the receiver waits on.
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t cluster_addr(const void* p, int cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(cta));
  return r;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
// the one local arrival, announcing the bytes the phase waits for
__device__ __forceinline__ void mbar_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t addr, int x, int y, int z, int w, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.s32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_s32(uint32_t addr, int x, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.s32 [%0], %1, [%2];" ::"r"(addr), "r"(x),
               "r"(bar)
               : "memory");
}
// Wait for phase 0 of an exchange barrier (cluster-scope acquire: the remote bytes are visible afterwards); false
// if it did not complete within XWAIT_LIMIT polls.
__device__ __forceinline__ bool mbar_wait0(uint64_t* b) {
  for (unsigned it = 0; it < XWAIT_LIMIT; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(b))
        : "memory");
    if (ok) return true;
  }
  return false;
}

// Walk a chunk sequence c, c + S, c + 2S, ... as (row, chunk-in-row) pairs without a division per step.
struct ChunkWalk {
  int q, w, sq, sw, cpr;
  __device__ __forceinline__ ChunkWalk(int c, int S, int cpr_) : cpr(cpr_) {
    q = c / cpr;
    w = c - q * cpr;
    sq = S / cpr;
    sw = S - sq * cpr;
  }
  __device__ __forceinline__ void next() {
    q += sq;
    w += sw;
    if (w >= cpr) {
      w -= cpr;
      ++q;
    }
  }
};

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
  uint16_t* s_cidx = reinterpret_cast<uint16_t*>(smem + L.cidx);
  int* s_tbl = reinterpret_cast<int*>(smem + L.tbl);
  int* s_red = reinterpret_cast<int*>(smem + L.red);
  int* s_wlo = reinterpret_cast<int*>(smem + L.wstat);
  int* s_whi = s_wlo + NW;
  int* s_wval = s_whi + NW;
  int* s_wmiss = s_wval + NW;
  int* s_misc = reinterpret_cast<int*>(smem + L.misc);
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(smem + L.mscr);   // token bitmap (short contexts)
  uint16_t* s_mbuf = reinterpret_cast<uint16_t*>(smem + L.mscr);   // sort buffers (long contexts)
  uint16_t* s_rank = reinterpret_cast<uint16_t*>(smem + L.rank);
  int32_t* s_bcnt = reinterpret_cast<int32_t*>(smem + L.bcnt);
  int32_t* s_blist = reinterpret_cast<int32_t*>(smem + L.blist);
  int32_t* s_vic = reinterpret_cast<int32_t*>(smem + L.vic);
  int32_t* s_xrow = reinterpret_cast<int32_t*>(smem + L.xrow);
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* vbar = xbar + 1;

  // Programmatic dependent launch: wait until the preceding kernel in the stream has completed and its writes
  // are visible, then let the next kernel start its launch while this one runs.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const int C = a.cluster;
  const int rank = blockIdx.x % C;
  // Clusters are (request b, layer group g); a group is a run of consecutive layers that share one selection, so
  // they hold identical metadata: each group resolves from its own first layer and updates only its own layers.
  const int nreq = (int)gridDim.x / (C * a.groups);
  const int b = (int)(blockIdx.x / C) % nreq, grp = (int)(blockIdx.x / C) / nreq;
  const int lgrp = (a.nlayers + a.groups - 1) / a.groups;
  const int l0 = grp * lgrp;
  const int nl = min(a.nlayers, l0 + lgrp) - l0;  // >= 1: the host makes at most nlayers groups
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, H = a.slots, ctx = a.ctx, R = a.row_bytes;
  // Each warp handles a contiguous run of selection entries in steps 2 and 3. The first entries of its run are
  // requested before anything else: the hit test waits on them and then on the token map, two round trips to
  // memory that the rest of the prologue overlaps.
  const int32_t* sel = a.topk + (size_t)b * k;
  const int wseg = ((k + NW * 32 - 1) / (NW * 32)) * 32;
  const int wbeg = min(k, warp * wseg);
  const int wend = min(k, wbeg + wseg);
  constexpr int RUN_STEP = 4 * 32;  // entries of a warp's run per iteration
  int32_t tn[4];
  auto load_sel = [&](int i0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * 32 + lane;
      tn[u] = i < wend ? ld_fresh(sel + i) : -1;
    }
  };
  load_sel(wbeg);
  const int32_t step = __ldcg(a.step) + a.begin;
  // On every way out: the last CTA of a step-beginning launch publishes the advanced step. Only the reads of the
  // old value must come first, and every thread of a CTA has read it (and used it) long before its thread 0 gets
  // here, past several barriers; later launches read the new value once this grid has completed.
  auto finish = [&]() {
    if (a.begin && tid == 0 && atomicAdd(a.done, 1) == (int)gridDim.x - 1) {
      *const_cast<int32_t*>(a.step) = step;
      *a.done = 0;
    }
  };
  int32_t* out = (a.out_slots && grp == 0) ? a.out_slots + (size_t)b * k : nullptr;  // identical in every group
  // The pool request of batch row b: req_ids[b] when the call maps rows to requests, else b. A row whose id is
  // out of range is rejected whole before any of the pool's memory is read (every CTA of the cluster reads the
  // same id and leaves here, before any barrier of the cluster).
  int rq = b;
  if (a.req_ids) {
    rq = ld_fresh(a.req_ids + b);
    if (rq < 0 || rq >= a.max_batch) {
      if (out)
        for (int i = tid; i < k; i += NT)
          if (((i >> 5) % C) == rank) out[i] = -1;
      if (rank == 0 && tid == 0) atomicOr(a.err, (int)HS_DEVERR_RANGE);
      finish();
      return;
    }
  }
  int32_t* t2s = a.tok2slot + (size_t)l0 * (size_t)a.meta_layer_ctx + (size_t)rq * ctx;
  int32_t* s2t = a.slot_tok + (size_t)l0 * (size_t)a.meta_layer_slots + (size_t)rq * H;
  int32_t* stp = a.slot_stamp + (size_t)l0 * (size_t)a.meta_layer_slots + (size_t)rq * H;
  unsigned long long* counters = a.counters + 4 * (size_t)l0;
  const uint8_t* src = a.src + (size_t)l0 * (size_t)a.src_layer_bytes + (size_t)rq * (size_t)a.src_req_stride;
  const int32_t* res = a.resident ? a.resident + (size_t)b * (size_t)a.resident_stride : nullptr;
  uint8_t* hot = a.hot + (size_t)l0 * (size_t)a.hot_layer_bytes + (size_t)rq * (size_t)H * (size_t)R;
  const int hwords = (H + 31) >> 5;
  const int cwords = (ctx + 31) >> 5;
  const int cpr = R >> 4;
  // Selection entries are owned by the CTAs of the cluster in runs of 32 (entry i belongs to CTA (i / 32) % C),
  // which write their metadata and out_slots. Row chunks go in blocks of BLK: block g belongs to CTA g % C.
  constexpr int BLK = 32 * COPY_UNROLL;
  auto owned = [&](int i) { return ((i >> 5) % C) == rank; };

  // 1. the slot metadata starts on its way to shared memory (asynchronous copies, waited for at the end of step
  //    2), and the bitmaps are cleared
  unsigned bad = 0;
  if ((H & 3) == 0) {  // per-request arrays start on 16-byte boundaries
    for (int c = tid; c < (H >> 2); c += NT) {
      cp_async16(s_stamp + 4 * c, stp + 4 * c);
      cp_async16(s_stok + 4 * c, s2t + 4 * c);
    }
  } else {
    for (int v = tid; v < H; v += NT) {
      cp_async4(s_stamp + v, stp + v);
      cp_async4(s_stok + v, s2t + v);
    }
  }
  cp_async_commit();
  if (tid < MISC_INTS) s_misc[tid] = 0;
  for (int w = tid; w < hwords; w += NT) s_hit[w] = 0u;
  if (BITMAP)
    for (int w = tid; w < cwords; w += NT) s_bits[w] = 0u;
  for (int x = tid; x < NBUCKET; x += NT) s_bcnt[x] = 0;
  if (tid == 0) {
    mbar_init(xbar, 1);
    mbar_init(vbar, 1);
    if (C > 1) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // every row of group B of every CTA of the cluster lands here (when there are misses to place)
    mbar_expect(xbar, (uint32_t)(C * (NW - GA_WARPS) * XROW * 4));
  }
  __syncthreads();
  // the exchange barriers exist before any CTA of the cluster sends to them (waited for after step 3)
  if (C > 1) cluster_arrive();

  // 2. hit test over this warp's run of entries: hits mark their slot, misses their token
  int nvalid = 0, nmiss = 0;
  for (int i0 = wbeg; i0 < wend; i0 += RUN_STEP) {
    int32_t t[4], s[4], r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) t[u] = tn[u];
    if (i0 + RUN_STEP < wend) load_sel(i0 + RUN_STEP);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * 32 + lane;
      const bool ok = t[u] >= 0 && t[u] < ctx;
      s[u] = ok ? __ldcg(t2s + t[u]) : -1;
      r[u] = (ok && res) ? ld_fresh(res + t[u]) : -1;
      if (i < wend) {
        s_sel[i] = t[u];
        if (t[u] >= ctx) bad |= HS_DEVERR_RANGE;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i >= wend) continue;
      int32_t sl = s[u];
      if (sl >= H) {
        bad |= HS_DEVERR_STATE;
        sl = -1;
      }
      if (sl < 0 && r[u] >= 0) sl = -2 - r[u];  // served in place from the HBM-resident tier
      s_slot[i] = sl;
      if (sl >= 0) {
        const uint32_t bit = 1u << (sl & 31);
        if (atomicOr(&s_hit[sl >> 5], bit) & bit) bad |= HS_DEVERR_DUP;
      } else if (sl <= -2) {
        // a repeated in-place token is caught here (bitmap; the bit is cleared again in step 3) or by a sort
        // of the in-place list, kept at the top of s_mpos (radix)
        if (BITMAP) {
          const uint32_t bit = 1u << (t[u] & 31);
          if (atomicOr(&s_bits[t[u] >> 5], bit) & bit) bad |= HS_DEVERR_DUP;
        } else {
          s_mpos[k - 1 - atomicAdd(&s_misc[MISC_NINP], 1)] = (uint16_t)i;
        }
      } else if (sl == -1 && t[u] >= 0 && t[u] < ctx) {
        if (BITMAP) {
          const uint32_t bit = 1u << (t[u] & 31);
          if (atomicOr(&s_bits[t[u] >> 5], bit) & bit) bad |= HS_DEVERR_DUP;
        }
        ++nmiss;
      }
      nvalid += t[u] >= 0 ? 1 : 0;
    }
  }
  nvalid = __reduce_add_sync(0xffffffffu, nvalid);
  nmiss = __reduce_add_sync(0xffffffffu, nmiss);
  if (lane == 0) {
    s_wval[warp] = nvalid;
    s_wmiss[warp] = nmiss;
  }
  cp_async_wait_all();
  __syncthreads();

  // 3. the misses in selection order (the same list in every CTA of the cluster)
  int m = 0, run = 0;
  for (int w = 0; w < NW; ++w) {
    const int x = s_wmiss[w];
    run += w < warp ? x : 0;
    m += x;
  }
  for (int base = wbeg; base < wend; base += 32) {
    const int i = base + lane;
    const bool f = i < wend && s_slot[i] == -1 && s_sel[i] >= 0 && s_sel[i] < ctx;
    if (BITMAP && i < wend && s_slot[i] <= -2) atomicAnd(&s_bits[s_sel[i] >> 5], ~(1u << (s_sel[i] & 31)));
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (f) s_mpos[run + __popc(bal & hs::lanemask_lt())] = (uint16_t)i;
    run += __popc(bal);
  }
  __syncthreads();
  if (C > 1) {
    cluster_wait();    // every CTA of the cluster runs, its exchange barriers initialised
    cluster_arrive();  // every read of the cluster-shared metadata by this CTA has returned its value
  }
  const int nchunk = m * cpr;  // 16-byte chunks of the rows; chunk c = chunk c % cpr of miss c / cpr
  const int nblk = (nchunk + BLK - 1) / BLK;
  // Blocks go to the CTAs in runs of RUN consecutive blocks (whole rows when rows span several blocks): run s
  // belongs to CTA s % C. Local block n of this CTA is global block (rank + C * (n / RUN)) * RUN + n % RUN.
  const int RUN = max(1, cpr / BLK);
  const int nrun = (nblk + RUN - 1) / RUN;
  const int my_runs = nrun > rank ? (nrun - rank + C - 1) / C : 0;
  const int my_blocks =
      my_runs ? (my_runs - 1) * RUN + min(RUN, nblk - (rank + C * (my_runs - 1)) * RUN) : 0;
  auto global_block = [&](int n) { return (rank + C * (n / RUN)) * RUN + n % RUN; };

  // 4. two warp groups at once
  uint4 pre[COPY_UNROLL];
  if (warp < GA_WARPS) {
    // A: the first wave of row loads (block number `warp` of this CTA), then the rank of every miss by token
    const Group g{0, GA_WARPS, 1};
    int* red = s_red;
    if (warp < my_blocks) {
      ChunkWalk cw(global_block(warp) * BLK + lane, 32, cpr);
#pragma unroll
      for (int u = 0; u < COPY_UNROLL; ++u) {
        if (cw.q < m)
          pre[u] = load_row_chunk<FROM_HOST>(src + (size_t)s_sel[s_mpos[cw.q]] * R + ((size_t)cw.w << 4));
        cw.next();
      }
    }
    if (m > 0) {
      // Rank of each miss among the misses by token, by a counting sort on the token's top bits: tokens fall into
      // at most NBUCKET buckets of 2^shift consecutive tokens; a miss's rank is the number of misses in earlier
      // buckets plus the smaller tokens in its own bucket (a handful); an equal token there is a repeat.
      const int shift = max(0, bits_of((unsigned)(ctx - 1)) - 11);
      for (int q = g.tid(); q < m; q += GA_THREADS) atomicAdd(&s_bcnt[s_sel[s_mpos[q]] >> shift], 1);
      g.sync();
      // buckets of this thread: a contiguous run of NBUCKET / 256 (all buckets are scanned: the unused ones
      // past nbk stay zero)
      constexpr int PER = NBUCKET / GA_THREADS;
      static_assert(PER % 4 == 0, "runs of whole 16-byte groups");
      int4 q4[PER / 4];
      int c = 0;
#pragma unroll
      for (int u = 0; u < PER / 4; ++u) {
        q4[u] = *reinterpret_cast<const int4*>(s_bcnt + g.tid() * PER + 4 * u);
        c += q4[u].x + q4[u].y + q4[u].z + q4[u].w;
      }
      int total;
      int start = hs::group_exclusive_scan(g, c, red, &total);
#pragma unroll
      for (int u = 0; u < PER / 4; ++u) {
        int4 o;
        o.x = start;
        o.y = o.x + q4[u].x;
        o.z = o.y + q4[u].y;
        o.w = o.z + q4[u].z;
        start = o.w + q4[u].w;
        *reinterpret_cast<int4*>(s_bcnt + g.tid() * PER + 4 * u) = o;
      }
      g.sync();
      // the tokens placed bucket by bucket; afterwards s_bcnt[x] is the end of bucket x (the start of x + 1)
      for (int q = g.tid(); q < m; q += GA_THREADS) {
        const int t = s_sel[s_mpos[q]];
        s_blist[atomicAdd(&s_bcnt[t >> shift], 1)] = t;
      }
      g.sync();
      for (int q = g.tid(); q < m; q += GA_THREADS) {
        const int pos = s_mpos[q];
        const int t = s_sel[pos], x = t >> shift;
        const int e = s_bcnt[x];
        int r = x ? s_bcnt[x - 1] : 0, eq = 0;
        for (int j = r; j < e; ++j) {
          const int y = s_blist[j];
          r += y < t;
          eq += y == t;
        }
        s_rank[pos] = (uint16_t)r;
        if (eq > 1) bad |= HS_DEVERR_DUP;
      }
    }
    if (!BITMAP && s_misc[MISC_NINP] > 1) {
      // repeated in-place tokens: sort the in-place list by token and compare neighbours
      const int ninp = s_misc[MISC_NINP];
      auto inp_tok = [&](int q) { return s_sel[s_mpos[k - 1 - q]]; };
      g.sync();  // the miss ranking no longer reads the sort buffers
      int n2 = 0;
      const uint16_t* order = hs::radix_sort(g, ninp, bits_of((unsigned)(ctx - 1)), s_mbuf, s_mbuf + k, inp_tok,
                                             [](int) { return true; }, s_tbl, red, &n2);
      for (int j = g.tid() + 1; j < ninp; j += GA_THREADS)
        if (inp_tok(order[j]) == inp_tok(order[j - 1])) bad |= HS_DEVERR_DUP;
    }
    if (tid == 0) s_misc[MISC_NEXT] = min(GA_WARPS, my_blocks);  // the first wave took blocks [0, this)
  } else {
    // B: victims in (stamp, slot) order, the m smallest keys among the slots not hit. The CTAs of the cluster
    //    split the slots: CTA r takes the r-th range, its warp w the w-th part of it, so segment r * 8 + w runs
    //    in ascending slot order.
    const Group g{GA_WARPS, NW - GA_WARPS, 2};
    int* red = s_red + RED_INTS;
    int ncand = 0;
    if (m > 0) {  // a call whose selection is all resident (a resolve after its prefetch) needs no victims
      auto cand = [&](int v) { return !(s_hit[v >> 5] & (1u << (v & 31))); };
      const int hc = ((H + C * g.size() - 1) / (C * g.size())) * g.size();  // slots per CTA
      const int hw = hc / g.nw;                                             // per warp, a multiple of 32
      const int sbeg = min(H, rank * hc + g.warp() * hw), send = min(H, sbeg + hw);
      const int sg = rank * g.nw + g.warp();
      // lanes of a run of 32 slots whose 5-bit bin is this lane's, from the run's bit planes of the bin
      auto bin_lanes = [&](unsigned part, unsigned p0, unsigned p1, unsigned p2, unsigned p3, unsigned p4) {
        return part & ((lane & 1) ? p0 : ~p0) & ((lane & 2) ? p1 : ~p1) & ((lane & 4) ? p2 : ~p2) &
               ((lane & 8) ? p3 : ~p3) & ((lane & 16) ? p4 : ~p4);
      };
      auto planes = [&](bool part, int x) {
        return bin_lanes(__ballot_sync(0xffffffffu, part), __ballot_sync(0xffffffffu, x & 1),
                         __ballot_sync(0xffffffffu, x & 2), __ballot_sync(0xffffffffu, x & 4),
                         __ballot_sync(0xffffffffu, x & 8), __ballot_sync(0xffffffffu, x & 16));
      };
      constexpr int U = 4;  // runs of 32 slots in flight per iteration
      // One pass over the segment: the candidates' stamp range and count, and (lane b) how many have
      // stamp % 32 == b. Once the range is known to span at most 32 stamps, these are the exact per-stamp counts.
      int smin = 0x7fffffff, smax = -1, nc = 0, cnt = 0;
      for (int base = sbeg; base < send; base += 32 * U) {
        int st[U];
        bool c[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = base + 32 * u + lane;
          c[u] = v < send && cand(v);
          st[u] = c[u] ? s_stamp[v] : 0;
          if (c[u]) {
            smin = min(smin, st[u]);
            smax = max(smax, st[u]);
            ++nc;
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) cnt += __popc(planes(c[u], st[u] & 31));
      }
      smin = (int)__reduce_min_sync(0xffffffffu, (unsigned)smin);  // stamps are >= 0
      smax = __reduce_max_sync(0xffffffffu, smax);
      nc = __reduce_add_sync(0xffffffffu, nc);
      // the segment's row goes to row sg of every CTA of the cluster (16-byte pieces, lanes 0-8)
      {
        const int p = lane < 8 ? lane : 0;
        const int x0 = __shfl_sync(0xffffffffu, cnt, 4 * p), x1 = __shfl_sync(0xffffffffu, cnt, 4 * p + 1),
                  x2 = __shfl_sync(0xffffffffu, cnt, 4 * p + 2), x3 = __shfl_sync(0xffffffffu, cnt, 4 * p + 3);
        int4 piece = lane < 8 ? make_int4(x0, x1, x2, x3) : make_int4(smin, smax, nc, 0);
        int32_t* row = s_xrow + sg * XROW + 4 * lane;
        if (C > 1) {
          if (lane < XROW / 4)
            for (int dst = 0; dst < C; ++dst)
              st_async_v4(cluster_addr(row, dst), piece.x, piece.y, piece.z, piece.w, cluster_addr(xbar, dst));
          if (!mbar_wait0(xbar)) s_misc[MISC_XFAIL] = 1;
          g.sync();  // every warp of the group takes the same branch below
        } else {
          if (lane < XROW / 4) *reinterpret_cast<int4*>(row) = piece;
          g.sync();
        }
      }
      const bool xfail = s_misc[MISC_XFAIL] != 0;
      if (xfail) bad |= HS_DEVERR_TIMEOUT;
      // the cluster's range and count (every warp reads the rows: lane j takes rows j and j + 32)
      const int nrows = C * g.nw;
      int gmin = 0x7fffffff, gmax = -1, gnc = 0;
#pragma unroll 2
      for (int j = lane; j < nrows; j += 32) {
        gmin = min(gmin, s_xrow[j * XROW + 32]);
        gmax = max(gmax, s_xrow[j * XROW + 33]);
        gnc += s_xrow[j * XROW + 34];
      }
      gmin = (int)__reduce_min_sync(0xffffffffu, (unsigned)gmin);
      gmax = __reduce_max_sync(0xffffffffu, gmax);
      gnc = __reduce_add_sync(0xffffffffu, gnc);
      ncand = gnc;
      if (m <= gnc && gnc == H && gmax == gmin && !xfail) {
        // no slot is hit and every slot has the same stamp (a cold start into empty caches): victim j is slot j
        for (int j = g.tid(); j < m; j += g.size()) s_vic[j] = j;
      } else if (m <= gnc && gmax - gmin <= 31 && !xfail) {
        // Stamp bin d = stamp - gmin < 32, lane d's counts in column (gmin + d) % 32. The bin totals and their
        // prefix give T, the bin holding position m - 1: bins below T are taken whole, bin T in slot order up to
        // m, at positions in (bin, segment, slot) order, which is (stamp, slot) order -- ties to the lowest slot.
        const int col = (gmin + lane) & 31;
        int before = 0, tot = 0;
#pragma unroll 8
        for (int j = 0; j < nrows; ++j) {
          const int x = s_xrow[j * XROW + col];
          before += j < sg ? x : 0;
          tot += x;
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        // T exists: every candidate lies in bins 0..31 and there are at least m of them
        const int T = __ffs(__ballot_sync(0xffffffffu, incl >= m)) - 1;
        int mybase = incl - tot + before;  // position of this segment's next slot of bin `lane`
        if (C > 1 && g.tid() == 0) mbar_expect(vbar, (uint32_t)(4 * m));
        for (int base = sbeg; base < send; base += 32 * U) {
          int d[U];
          unsigned mine[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = base + 32 * u + lane;
            d[u] = (v < send && cand(v)) ? s_stamp[v] - gmin : 32;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) mine[u] = planes(d[u] <= T, d[u]);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int from = d[u] <= T ? d[u] : 0;
            const unsigned peers = __shfl_sync(0xffffffffu, mine[u], from);
            const int at = __shfl_sync(0xffffffffu, mybase, from);
            if (d[u] <= T) {
              const int pos = at + __popc(peers & hs::lanemask_lt());
              if (d[u] < T || pos < m) {
                const int v = base + 32 * u + lane;
                if (C > 1)
                  for (int dst = 0; dst < C; ++dst)
                    st_async_s32(cluster_addr(s_vic + pos, dst), v, cluster_addr(vbar, dst));
                else
                  s_vic[pos] = v;
              }
            }
            mybase += __popc(mine[u]);
          }
        }
        if (C > 1) {
          if (!mbar_wait0(vbar)) bad |= HS_DEVERR_TIMEOUT;
        }
      } else if (m <= gnc && !xfail) {
        // the candidates span more than 32 stamps: every CTA sorts all of them (stable LSD on stamp - gmin)
        int n2 = 0;
        const uint16_t* order = hs::radix_sort(
            g, H, bits_of((unsigned)(gmax - gmin)), s_cidx, s_cidx + H, [&](int v) { return s_stamp[v] - gmin; },
            cand, s_tbl, red, &n2, m);
        for (int j = g.tid(); j < m; j += g.size()) s_vic[j] = order[j];
      }
    }
    if (g.tid() == 0) s_misc[MISC_NCAND] = ncand;
  }
  if (bad) atomicOr(&s_misc[MISC_BAD], (int)bad);
  __syncthreads();
  bad = (unsigned)s_misc[MISC_BAD] | (m > s_misc[MISC_NCAND] ? HS_DEVERR_STATE : 0u);

  if (bad) {
    // a rejected row changes no metadata, so no cluster barrier is needed
    if (out)
      for (int i = tid; i < k; i += NT)
        if (owned(i)) out[i] = -1;
    if (rank == 0 && tid == 0) atomicOr(a.err, (int)bad);
    finish();
    return;
  }

  // victim of the miss at selection entry i
  auto victim_of = [&](int i, int) -> int { return s_vic[s_rank[i]]; };
  auto store_chunk_to = [&](uint8_t* dst_hot, int q, int w, const uint4& val) {
    const int i = s_mpos[q];
    *reinterpret_cast<uint4*>(dst_hot + (size_t)victim_of(i, s_sel[i]) * R + ((size_t)w << 4)) = val;
  };
  auto store_chunk = [&](int q, int w, const uint4& val) { store_chunk_to(hot, q, w, val); };

  // this CTA's row blocks past the first wave, one per warp at a time from a shared counter; with several
  // layers, local block n is block n % my_blocks of layer n / my_blocks
  auto copy_rows = [&]() {
    while (true) {
      int n = 0;
      if (lane == 0) n = atomicAdd(&s_misc[MISC_NEXT], 1);
      n = __shfl_sync(0xffffffffu, n, 0);
      if (n >= my_blocks * nl) break;
      const int l = n / my_blocks;
      const int nb = n - l * my_blocks;
      const uint8_t* src_l = src + (size_t)l * (size_t)a.src_layer_bytes;
      uint8_t* hot_l = hot + (size_t)l * (size_t)a.hot_layer_bytes;
      uint4 v[COPY_UNROLL];
      ChunkWalk cw(global_block(nb) * BLK + lane, 32, cpr);
#pragma unroll
      for (int u = 0; u < COPY_UNROLL; ++u) {
        if (cw.q < m) v[u] = load_row_chunk<FROM_HOST>(src_l + (size_t)s_sel[s_mpos[cw.q]] * R + ((size_t)cw.w << 4));
        cw.next();
      }
      ChunkWalk cs(global_block(nb) * BLK + lane, 32, cpr);
#pragma unroll
      for (int u = 0; u < COPY_UNROLL; ++u) {
        if (cs.q < m) store_chunk_to(hot_l, cs.q, cs.w, v[u]);
        cs.next();
      }
    }
  };

  int nevict = 0;
  if (warp >= GA_WARPS) {
    // B: rows past the first wave, at once (hot-buffer slots are read by no other CTA, so no barrier)
    copy_rows();
    if (C > 1) cluster_wait();
  } else {
    // A: 5. per owned selection entry, once every CTA of the cluster has read the metadata: hits are
    //    stamped, a miss of rank j takes victim j
    if (C > 1) cluster_wait();
    // this CTA's runs of 32 entries are rank, rank + C, ...: warp w takes runs w, w + 8, ... of them
    for (int i = (rank + C * warp) * 32 + lane; i < k; i += C * GA_WARPS * 32) {
      const int32_t t = s_sel[i];
      const int32_t s = s_slot[i];
      if (s >= 0) {
        for (int l = 0; l < nl; ++l) stp[(size_t)l * (size_t)a.meta_layer_slots + s] = step;
        if (out) out[i] = s;
      } else if (t < 0 || s <= -2) {
        if (out) out[i] = t < 0 ? -1 : s;  // padding, or a row served in place (-2 - its pool row)
      } else {
        const int32_t v = victim_of(i, t);
        const int32_t u = s_stok[v];
        if (u >= 0) ++nevict;
        for (int l = 0; l < nl; ++l) {
          int32_t* t2s_l = t2s + (size_t)l * (size_t)a.meta_layer_ctx;
          const size_t sl = (size_t)l * (size_t)a.meta_layer_slots;
          if (u >= 0) t2s_l[u] = -1;
          t2s_l[t] = v;
          s2t[sl + v] = t;
          stp[sl + v] = step;
        }
        if (out) out[i] = v;
      }
    }
    // 6. the first wave lands in the victims' slots, then this group joins the copy
    if (warp < my_blocks) {
      ChunkWalk cw(global_block(warp) * BLK + lane, 32, cpr);
#pragma unroll
      for (int u = 0; u < COPY_UNROLL; ++u) {
        if (cw.q < m) store_chunk(cw.q, cw.w, pre[u]);
        cw.next();
      }
    }
    copy_rows();
  }

  // counters
  nevict = __reduce_add_sync(0xffffffffu, nevict);
  if (lane == 0 && nevict)
    for (int l = 0; l < nl; ++l) atomicAdd(counters + 4 * l + 2, (unsigned long long)nevict);
  if (rank == 0 && tid == 0) {
    int nv = 0;
    for (int w = 0; w < NW; ++w) nv += s_wval[w];
    for (int l = 0; l < nl; ++l) {
      atomicAdd(counters + 4 * l + 0, (unsigned long long)(nv - m));
      atomicAdd(counters + 4 * l + 1, (unsigned long long)m);
      atomicAdd(counters + 4 * l + 3, (unsigned long long)m * (unsigned long long)R);
    }
  }
  finish();
}

// Gather rows by index, the read a sparse-attention kernel makes: row i of request b goes to
// dst[(b * k + i) * row_bytes]; an index < 0 or >= limit gives a zero row. Rows of request b start at
// base + b * req_stride. 16-byte chunks, COPY_UNROLL loads in flight per thread.
template <bool FROM_HOST>
__global__ void hs_gather_kernel(const uint8_t* __restrict__ base, int64_t req_stride, int row_bytes,
                                 const int32_t* __restrict__ idx, int k, int rows, int limit,
                                 uint8_t* __restrict__ dst) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int cpr = row_bytes >> 4;
  const long long n = (long long)rows * cpr;
  const long long nth = (long long)gridDim.x * blockDim.x;
  for (long long c0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; c0 < n; c0 += nth * COPY_UNROLL) {
    uint4 v[COPY_UNROLL];
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u) {
      const long long c = c0 + u * nth;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (c < n) {
        const int r = (int)(c / cpr);
        const int w = (int)(c - (long long)r * cpr);
        const int t = ld_fresh(idx + r);
        if (t >= 0 && t < limit) {
          const uint8_t* p = base + (size_t)(r / k) * (size_t)req_stride + (size_t)t * row_bytes + ((size_t)w << 4);
          v[u] = FROM_HOST ? load_row_chunk_host(p) : __ldcg(reinterpret_cast<const uint4*>(p));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < COPY_UNROLL; ++u) {
      const long long c = c0 + u * nth;
      if (c < n) *reinterpret_cast<uint4*>(dst + ((size_t)c << 4)) = v[u];
    }
  }
}

// Does nothing but take part in programmatic dependent launch: launched with a resolve's exact configuration, it
// measures the fixed cost of the launch itself (the floor under a resolve step).
__global__ void __launch_bounds__(NT, 1) hs_empty_kernel(const ResolveArgs) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
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

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool geometry_ok(const hs_pool_desc* d) {
  if (!d) return false;
  if (d->layers < 1 || d->max_batch < 1 || d->ctx < 1 || d->slots < 1 || d->topk_max < 1) return false;
  if (d->topk_max > d->slots || d->slots > 65535) return false;
  if (d->row_bytes <= 0 || (d->row_bytes & 15)) return false;
  // the kernel numbers the 16-byte chunks of one request-layer's misses with int
  if ((int64_t)d->topk_max * (d->row_bytes >> 4) > (int64_t)0x7fffffff - (int64_t)COPY_UNROLL * 2 * 8 * 512)
    return false;
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

#ifndef HS_PREFETCH_TARGET
// CTAs a prefetch aims for. A prefetch runs beside the layer's own work: half the resolve's footprint leaves that
// work its SMs while still keeping enough loads in flight for the link.
#define HS_PREFETCH_TARGET 32
#endif

int pick_cluster(const hs_pool* p, int batch, bool prefetch) {
  // Enough CTAs to keep the host link (or HBM, in no-IO mode) busy -- the link saturates with a few dozen
  // SMs -- without spilling the grid into a second wave.
  const int target = p->noio ? p->resident : (prefetch ? HS_PREFETCH_TARGET : 64);
  int c = 1;
  while (c < p->max_cluster && batch * c < target && batch <= p->max_active[2 * c]) c <<= 1;
  return c;
}

int launch_resolve(hs_pool* p, int32_t layer, int32_t batch, const int32_t* topk, int32_t k, int32_t* out,
                   cudaStream_t s, int32_t nlayers = 1, const int32_t* resident = nullptr,
                   int64_t resident_stride = 0, bool empty = false, const int32_t* req_ids = nullptr) {
  if (!p || layer < 0 || nlayers < 1 || layer > p->d.layers - nlayers || batch < 0 || batch > p->d.max_batch ||
      k < 0 || k > p->d.topk_max)
    return HS_ERR_INVALID_ARG;
  if (batch == 0 || k == 0) return HS_OK;
  if (!topk && !empty) return HS_ERR_INVALID_ARG;
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
  a.done = p->err + 1;  // the header's third word
  a.begin = 0;
  if (!empty && p->begin_pending) {
    a.begin = p->begin_pending;
    p->begin_pending = 0;
  }
  a.src = p->src + (size_t)layer * (size_t)p->d.host_layer_stride;
  a.src_req_stride = p->d.host_req_stride ? p->d.host_req_stride : (int64_t)p->d.ctx * p->d.row_bytes;
  a.hot = static_cast<uint8_t*>(p->d.hot_buf) + rl0 * (size_t)p->d.slots * (size_t)p->d.row_bytes;
  a.k = k;
  a.ctx = p->d.ctx;
  a.slots = p->d.slots;
  a.row_bytes = p->d.row_bytes;
  a.cluster = pick_cluster(p, batch, out == nullptr && !empty);
  a.nlayers = nlayers;
  a.groups = 1;
  if (nlayers > 1) {
    // Several layers sharing one selection: the layers are split into groups, one cluster per (request, group),
    // as many groups as the device holds clusters of that size at once, so that the row copies of all the layers
    // use the whole device. The cluster size is the largest whose grid reaches 80 % of the largest such grid
    // (bigger clusters split the victim choice finer).
    auto groups_for = [&](int c) {
      const int fit = c > 1 ? p->max_active[c] : p->resident;
      return fit >= batch ? std::min(nlayers, fit / batch) : 0;
    };
    int most = 0;
    for (int c = 1; c <= p->max_cluster; c <<= 1) most = std::max(most, batch * c * groups_for(c));
    for (int c = p->max_cluster; c >= 1; c >>= 1) {
      const int g = groups_for(c);
      if (g > 0 && 5 * batch * c * g >= 4 * most) {
        a.cluster = c;
        a.groups = g;
        break;
      }
    }
  }
  a.resident = resident;
  a.resident_stride = resident_stride;
  a.req_ids = req_ids;
  a.max_batch = p->d.max_batch;
  a.meta_layer_ctx = (int64_t)p->d.max_batch * p->d.ctx;
  a.meta_layer_slots = (int64_t)p->d.max_batch * p->d.slots;
  a.src_layer_bytes = p->d.host_layer_stride;
  a.hot_layer_bytes = (int64_t)p->d.max_batch * p->d.slots * p->d.row_bytes;

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(batch * a.cluster * a.groups), 1, 1);
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
  if (empty)
    e = cudaLaunchKernelEx(&cfg, hs_empty_kernel, a);
  else if (p->noio)
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
          cudaSuccess ||
      cudaFuncSetAttribute(hs_empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
    return HS_ERR_CUDA;

  hs_pool* p = new (std::nothrow) hs_pool;
  if (!p) return HS_ERR_NO_MEMORY;
  p->d = *desc;
  p->lay = lay;
  p->begin_pending = 0;
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
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hs_resolve_kernel<true, true>, NT, smem) !=
          cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  p->resident = per_sm * sms;
  for (int c = 0; c <= MAX_CLUSTER; ++c) p->max_active[c] = 0;
  p->max_active[1] = p->resident;
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
    p->max_active[c] = n;
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
  pool->begin_pending = 0;
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

int hs_step_begin_fused(hs_pool* pool) {
  if (!pool) return HS_ERR_INVALID_ARG;
  ++pool->begin_pending;
  return HS_OK;
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

int hs_resolve_ids(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* req_ids, const int32_t* topk_idx,
                   int32_t k, int32_t* out_slots, hs_stream_t stream) {
  if (batch > 0 && k > 0 && (!out_slots || !req_ids)) return HS_ERR_INVALID_ARG;
  return launch_resolve(pool, layer, batch, topk_idx, k, out_slots, reinterpret_cast<cudaStream_t>(stream), 1,
                        nullptr, 0, false, req_ids);
}

int hs_prefetch_ids(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* req_ids, const int32_t* topk_idx,
                    int32_t k, hs_stream_t stream) {
  if (batch > 0 && k > 0 && !req_ids) return HS_ERR_INVALID_ARG;
  return launch_resolve(pool, layer, batch, topk_idx, k, nullptr, reinterpret_cast<cudaStream_t>(stream), 1,
                        nullptr, 0, false, req_ids);
}

static int launch_gather(hs_pool* p, int32_t layer, int32_t batch, const int32_t* idx, int32_t k, void* dst,
                         hs_stream_t stream, bool history) {
  if (!p || layer < 0 || layer >= p->d.layers || batch < 0 || batch > p->d.max_batch || k < 0 ||
      k > p->d.topk_max)
    return HS_ERR_INVALID_ARG;
  if (batch == 0 || k == 0) return HS_OK;
  if (!idx || !dst || (reinterpret_cast<uintptr_t>(dst) & 15)) return HS_ERR_INVALID_ARG;
  const int rows = batch * k;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  const long long chunks = (long long)rows * (p->d.row_bytes >> 4);
  const long long per_cta = (long long)NT * COPY_UNROLL;
  cfg.gridDim = dim3((unsigned)std::min<long long>((chunks + per_cta - 1) / per_cta, 2LL * p->num_sms), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  uint8_t* out = static_cast<uint8_t*>(dst);
  cudaError_t e;
  if (history) {
    const uint8_t* base = p->src + (size_t)layer * (size_t)p->d.host_layer_stride;
    const int64_t rs = p->d.host_req_stride ? p->d.host_req_stride : (int64_t)p->d.ctx * p->d.row_bytes;
    e = p->noio ? cudaLaunchKernelEx(&cfg, hs_gather_kernel<false>, base, rs, p->d.row_bytes, idx, k, rows,
                                     p->d.ctx, out)
                : cudaLaunchKernelEx(&cfg, hs_gather_kernel<true>, base, rs, p->d.row_bytes, idx, k, rows,
                                     p->d.ctx, out);
  } else {
    const size_t hrl = (size_t)p->d.slots * (size_t)p->d.row_bytes;
    const uint8_t* base = static_cast<const uint8_t*>(p->d.hot_buf) + (size_t)layer * (size_t)p->d.max_batch * hrl;
    e = cudaLaunchKernelEx(&cfg, hs_gather_kernel<false>, base, (int64_t)hrl, p->d.row_bytes, idx, k, rows,
                           p->d.slots, out);
  }
  return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_gather(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* out_slots, int32_t k, void* dst,
              hs_stream_t stream) {
  return launch_gather(pool, layer, batch, out_slots, k, dst, stream, false);
}

int hs_gather_history(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* topk_idx, int32_t k, void* dst,
                      hs_stream_t stream) {
  return launch_gather(pool, layer, batch, topk_idx, k, dst, stream, true);
}

int hs_resolve_shared(hs_pool* pool, int32_t layer0, int32_t nlayers, int32_t batch, const int32_t* topk_idx,
                      int32_t k, int32_t* out_slots, hs_stream_t stream) {
  if (batch > 0 && k > 0 && !out_slots) return HS_ERR_INVALID_ARG;
  return launch_resolve(pool, layer0, batch, topk_idx, k, out_slots, reinterpret_cast<cudaStream_t>(stream),
                        nlayers);
}

int hs_resolve_tiered(hs_pool* pool, int32_t layer, int32_t batch, const int32_t* topk_idx, int32_t k,
                      const int32_t* resident_row, int64_t resident_stride, int32_t* out_slots,
                      hs_stream_t stream) {
  if (batch > 0 && k > 0 && (!out_slots || !resident_row)) return HS_ERR_INVALID_ARG;
  if (!pool || resident_stride < (int64_t)pool->d.ctx) return HS_ERR_INVALID_ARG;
  return launch_resolve(pool, layer, batch, topk_idx, k, out_slots, reinterpret_cast<cudaStream_t>(stream), 1,
                        resident_row, resident_stride);
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

int hs_probe_launch(hs_pool* pool, int32_t layer, int32_t nlayers, int32_t batch, int32_t k, hs_stream_t stream) {
  return launch_resolve(pool, layer, batch, nullptr, k, nullptr, reinterpret_cast<cudaStream_t>(stream), nlayers,
                        nullptr, 0, true);
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
  for (int r = 0; r <= iters && rc == HS_OK; ++r) {  // iteration 0 warms up
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
    case HS_ERR_TOO_LARGE: return "request larger than the fixed device scratch of hs_probe_link_static (16 MiB)";
    default: return "unknown error";
  }
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------------------------
// Link probe that allocates nothing (hs_probe_link_static)
// ------------------------------------------------------------------------------------------------------------------

// Its device scratch: the copy's destination and the read kernel's sink (the first HS_STATIC_PROBE_MAX bytes), then
// four clock stamps. A module global, so every device that loads this library holds it until the process exits.
constexpr size_t HS_STATIC_PROBE_MAX = (size_t)16 << 20;
static __device__ __align__(256) unsigned char hs_static_probe_scratch[HS_STATIC_PROBE_MAX + 256];

namespace {

__global__ void hs_clock_stamp_kernel(unsigned long long* dst) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  *dst = t;
}

// Device address of the scratch on the current device, looked up once per device (a host-side name of a
// __device__ array is not a device address).
std::mutex g_static_probe_mu;
void* g_static_probe_addr[64];

int static_probe_scratch(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_static_probe_mu);
  if (!g_static_probe_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, hs_static_probe_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_static_probe_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_static_probe_addr[dev]);
  return HS_OK;
}

}  // namespace

extern "C" int hs_probe_link_static(const void* host, size_t bytes, int32_t iters, hs_stream_t stream,
                                    double* zero_copy_gbs, double* memcpy_gbs) {
  if (!host || bytes < 16 || (bytes & 15) || iters < 1 || !zero_copy_gbs || !memcpy_gbs ||
      (reinterpret_cast<uintptr_t>(host) & 15))
    return HS_ERR_INVALID_ARG;
  if (bytes > HS_STATIC_PROBE_MAX) return HS_ERR_TOO_LARGE;
  const void* dhost = mapped_host_ptr(host);
  if (!dhost) return HS_ERR_NOT_MAPPED;
  unsigned char* scratch = nullptr;
  int rc = static_probe_scratch(&scratch);
  if (rc != HS_OK) return rc;
  unsigned long long* stamps = reinterpret_cast<unsigned long long*>(scratch + HS_STATIC_PROBE_MAX);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev_id = 0, sms = 0;
  if (cudaGetDevice(&dev_id) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_id) != cudaSuccess)
    return HS_ERR_CUDA;
  // The same two transfers as hs_probe_link, timed by device clock stamps written into the scratch (no events).
  unsigned long long best_zc = ~0ull, best_cp = ~0ull;
  for (int r = 0; r <= iters; ++r) {  // iteration 0 warms up
    hs_clock_stamp_kernel<<<1, 1, 0, s>>>(stamps + 0);
    hs_probe_read_kernel<<<2 * sms, 512, 0, s>>>(static_cast<const uint8_t*>(dhost), bytes >> 4,
                                                  reinterpret_cast<unsigned*>(scratch));
    hs_clock_stamp_kernel<<<1, 1, 0, s>>>(stamps + 1);
    hs_clock_stamp_kernel<<<1, 1, 0, s>>>(stamps + 2);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(scratch, host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return HS_ERR_CUDA;
    hs_clock_stamp_kernel<<<1, 1, 0, s>>>(stamps + 3);
    unsigned long long t[4];
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(t, stamps, sizeof(t), cudaMemcpyDeviceToHost) != cudaSuccess)
      return HS_ERR_CUDA;
    if (r) {
      best_zc = std::min(best_zc, t[1] - t[0]);
      best_cp = std::min(best_cp, t[3] - t[2]);
    }
  }
  *zero_copy_gbs = (double)bytes / (double)std::max(best_zc, 1ull);  // bytes per ns = GB/s
  *memcpy_gbs = (double)bytes / (double)std::max(best_cp, 1ull);
  return HS_OK;
}
