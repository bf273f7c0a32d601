// Sparse MLA decode attention over the rows a resolve selected, sm_103a (tcgen05 tensor cores, TMEM accumulators).
//
// The resolver exists so that a sparse-attention kernel reads the selected KV rows from the GPU hot buffer
// instead of the full history, with model outputs unchanged ("HiSparse" paper, Abstract; the "Hybrid HiSparse"
// knowledge card builds on Sparse MLA). This is that consumer for one decode step of multi-head latent attention
// in its absorbed form: each row is 576 bf16 values (the 512-dimensional latent, then the 64-dimensional rotary
// key), 128 query heads each have a 576-dimensional query, and per request
//
//     s[h][i] = sm_scale * q[h] . row_i,   out[h] = sum_i softmax_i(s[h]) * row_i[0:512],   lse[h] = log sum_i e^s
//
// over the valid selected rows. The same kernel reads the rows either through a slot list (the hot buffer, plus
// rows still held in the ordinary HBM pool for entries -2 - row) or by token from the full history, so the two
// results are bit-identical whenever the rows are.
//
// A pair of CTAs splits the score GEMM's 576 columns: CTA 0 of the pair holds columns 0..255 of Q and of every
// selected row, CTA 1 columns 256..575. Each computes partial scores over its columns on the tensor cores, sends
// them to the other through distributed shared memory, and adds the other's. Both then hold the same S (addition
// commutes), run the same softmax, and each multiplies P by its own value half (columns 0..255 or 256..511, which
// lie within its columns). No score work is repeated. Each CTA keeps its columns of Q in tensor memory, as the
// score GEMM's A operand, which leaves shared memory to four key stages.
// A request's keys are split in two as well (two pairs, a cluster of four CTAs) whenever every request's cluster
// fits on the device at once: each pair runs the softmax over its half of the key blocks, and each merges half of
// the heads (flash-decoding's split-K merge, inside one cluster): for the other heads a pair writes its normalised
// output to `out` and its (max, normaliser) per head into the other pair's shared memory, and after a cluster
// barrier merges its own heads with what the other pair left. A pair's time is a chain of dependent steps per key
// block, not a bandwidth, so two pairs per request halve it.
// Warp roles per CTA:
//   warps 0-7   softmax: warp w owns heads 32 (w % 4) .. +31 (TMEM lanes of its quarter) for the keys of its half
//               w / 4 of every 64-key block; the two threads of a head agree on the block maximum through shared
//               memory and an mbarrier, and each sums its own weights;
//   warp 8      lane 0 issues every tcgen05.mma (and warp 8 allocates / frees the tensor memory);
//   warps 9-16  load the CTA's columns of the selected rows into shared memory with cp.async (zero rows for
//               padding), 64 rows per block, two warps per key stage (one per half of the block's keys),
//               prefetching each stage's next rows into L2;
//   warp 17     hands the score-exchange buffer back to the peer once it has been read.
// Shared memory: four key stages (64 rows each), one P buffer and one exchange buffer, in the no-swizzle
// interleaved layout: element (row r, column c) at (r/8)*G + (c/8)*128 +
// (r%8)*16 + (c%8)*2, where G is the byte size of an 8-row group (one spare 128-byte slot included). A key stage
// serves the score GEMM as a K-major operand (rows = keys) and the value GEMM as an MN-major operand (the same
// bytes read with the two strides exchanged).
// Tensor memory (512 columns): this CTA's columns of Q (two bf16 per column, up to 160 columns), one 64-column
// score buffer at column 192, and the 256-column output half at column 256.
// Per key block j: partial S = Q K^T (16 or 20 MMAs of 128x64x16, A from tensor memory) into the score buffer; the
// softmax threads read it, store it into the peer's exchange buffer with st.async (completing the bytes the peer's
// barrier expects), wait for the peer's part, and update the running max m (raised only when a block's maximum exceeds
// it by more than 8 in log2 units, which bounds P and O by 2^8 and makes the rescale of O rare); they write
// P = 2^(s - m) rounded to bf16 into the P buffer once the value GEMM of block j-1 has read it, and sum the
// rounded values; then O += P V (four 128x256x16 MMAs). The score GEMM of block j+1 starts as soon as the
// softmax threads have read block j's scores, and overlaps the rest of block j's softmax. The output leaves
// through a shared tile in whole 128-byte row segments. mbarriers order the roles,
// within the CTA and across the pair; every wait is bounded: on running out
// it sets an abort flag that ends every role and the HS_DEVERR_TIMEOUT bit of the pool's error word, after the
// issued MMAs and copies have drained. Cluster barriers at the start and the end keep each CTA's shared memory
// alive while the other may still reach it.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/hs.h"
#include "hs_pool.hpp"

namespace {

constexpr int HEADS = 128;
constexpr int DQK = 576;
constexpr int DV = 512;
constexpr int DV_HALF = DV / 2;
constexpr int ROW_BYTES = DQK * 2;
constexpr int KB = 64;       // keys per block (the N of the score GEMM)
constexpr int KH = KB / 2;   // keys of a block per softmax thread (two threads per head)
constexpr int NSTAGE = 4;    // key stages
constexpr int NPB = 1;       // P buffers
// Score-GEMM columns of each CTA of a request's pair: CTA 0 the first DSPLIT (its value half), CTA 1 the rest,
// which contain its value half (columns 256..511).
constexpr int DSPLIT = 256;
constexpr int MAX_NDIM = DQK - DSPLIT;
// An 8-row group of a CTA's columns holds its 16-byte chunks at 128-byte spacing plus one spare 128-byte slot, so
// that successive groups do not start at power-of-two distances.
constexpr int MAX_GROUP = (MAX_NDIM / 8 + 1) * 128;
constexpr int STAGE_BYTES = (KB / 8) * MAX_GROUP;
constexpr int P_GROUP = (KB / 8) * 128;    // bytes of one 8-head group of P (128 x KB)
constexpr int P_BYTES = HEADS * KB * 2;
constexpr int X_BYTES = HEADS * KB * 4;    // the peer's partial scores of one block, fp32
// Warp roles: softmax warps 0-7 (warp w: heads 32 (w % 4) .. +31, the block's keys KH (w / 4) .. +KH-1), the MMA
// issuer, loader warps (two per key stage), the exchange warp.
constexpr int SOFTMAX_WARPS = 8, SOFTMAX_THREADS = SOFTMAX_WARPS * 32, MMA_WARP = 8, LOAD_WARP0 = 9;
constexpr int STAGE_WARPS = 2;             // loader warps per key stage (one per half of the block's keys)
constexpr int LOAD_WARPS = NSTAGE * STAGE_WARPS;
constexpr int XCHG_WARP = LOAD_WARP0 + LOAD_WARPS;  // hands the exchange buffer back to the peer
constexpr int NTHREADS = (XCHG_WARP + 1) * 32;
// Tensor memory: this CTA's columns of Q (the score GEMM's A operand, two bf16 per 32-bit column: at most 160
// columns), the score buffer (KB columns) and the output half (256 columns).
constexpr uint32_t TMEM_COLS = 512, TMEM_Q = 0, TMEM_S = 192, TMEM_O = 256;
static_assert(TMEM_Q + MAX_NDIM / 2 <= TMEM_S && TMEM_S + KB <= TMEM_O, "tensor memory columns");
constexpr unsigned WAIT_LIMIT = 1u << 20;  // try_wait rounds (each may suspend briefly) before a wait gives up

constexpr int OFF_K = 0;
constexpr int OFF_P = OFF_K + NSTAGE * STAGE_BYTES;
constexpr int OFF_X = OFF_P + NPB * P_BYTES;       // one exchange buffer
constexpr int OFF_KEY = OFF_X + X_BYTES;           // row pointers of each stage: [NSTAGE][KB]
// mbarriers: kfull[NSTAGE] kempty[NSTAGE] sfull sempty pfull[NPB] pdone[NPB] odone drain xfull xempty xread tdone
// pmx[4] (the two softmax warps of a head quarter agreeing on the block maximum) qready (Q is in tensor memory)
constexpr int NBAR = 2 * NSTAGE + 2 + 2 * NPB + 2 + 3 + 1 + 4 + 1;
constexpr int OFF_BAR = OFF_KEY + NSTAGE * KB * 8;
// TMEM address, abort flag, per-stage stop flags, per-stage masks of the keys with a row (one word per half)
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_PMAX = (OFF_MISC + 8 + 4 * NSTAGE + 8 * NSTAGE + 15) & ~15;  // [2 parities][2 halves][HEADS]
// (m, l) per head from the CTA of the other key half, for the heads this CTA merges
constexpr int OFF_COMB = OFF_PMAX + 2 * 2 * HEADS * 4;
constexpr int SMEM_BYTES = OFF_COMB + HEADS * 8;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
static_assert(SOFTMAX_WARPS * 32 * 36 * 4 <= NSTAGE * STAGE_BYTES, "output tiles of the softmax warps fit the stages");
static_assert(KB == 2 * 32 && STAGE_WARPS >= 2, "one lane of the stage's first two warps per key of a block");

struct MlaArgs {
  const uint16_t* q;        // bf16 [batch][HEADS][DQK]
  const int32_t* idx;       // [batch][k]: slots (mode 0) or tokens (mode 1)
  int32_t k;
  int32_t mode;             // 0: slot list into `rows` (+ resident rows); 1: tokens into `rows`
  const uint8_t* rows;      // request 0's rows of this layer
  int64_t req_stride;       // bytes between requests in `rows`
  int32_t limit;            // valid indices into `rows` are 0 .. limit-1
  const uint8_t* resident;  // mode 0: rows for entries -2 - r, or nullptr
  int64_t resident_count;
  float scale_log2;         // sm_scale * log2(e)
  int32_t nsplit;           // 1 or 2 key halves per request (clusters of 2 * nsplit CTAs)
  float* out;               // [batch][HEADS][DV]
  float* lse;               // [batch][HEADS]
  int32_t* err;
  uint32_t wait_limit;      // polling rounds before a role's wait gives up (WAIT_LIMIT unless a test lowers it)
  int32_t stall;            // test hook: the issuer first waits on a barrier that nothing completes
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ int32_t ld_fresh(const int32_t* p) {
  int32_t v;
  asm("ld.global.cv.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// fetch a row into L2 ahead of its copy (bytes: multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// shared-memory writes of this thread become visible to the tensor cores' (async proxy) reads
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void bar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_test(uint64_t* b, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of the given parity.
__device__ __forceinline__ bool bar_poll(uint64_t* b, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of the given parity; false once the abort flag is set or after `limit` rounds (which sets
// it).
__device__ __forceinline__ bool bar_wait(uint64_t* b, unsigned parity, volatile int* abort_flag,
                                         unsigned limit = WAIT_LIMIT) {
  for (unsigned it = 0; it < limit; ++it) {
    if (bar_test(b, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// The pair's peer CTA: its copy of a shared-memory address, remote stores and remote arrivals.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(su32(p)), "r"(rank));
  return r;
}
// asynchronous remote store; its 16 bytes count toward the transaction bytes the peer's barrier expects
__device__ __forceinline__ void st_peer_async_v4(uint32_t addr, float a, float b, float c, float d, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(mbar)
               : "memory");
}
// arrive on a local barrier and expect `bytes` transaction bytes in its current phase
__device__ __forceinline__ void bar_arrive_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// 2^x by the hardware approximation (relative error far below the bf16 rounding that follows)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void bar_arrive_peer(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// a wait whose arrivals come from the peer (cluster-scope acquire makes its stores visible)
__device__ __forceinline__ bool bar_wait_cluster(uint64_t* b, unsigned parity, volatile int* abort_flag,
                                                 unsigned limit) {
  for (unsigned it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void st_peer_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: start, leading-dimension and stride-dimension byte offsets.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor: bf16 x bf16 -> f32, M x N, operand majors (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// The same with the A operand in tensor memory (M lanes; a 16-wide K chunk of bf16 is 8 columns).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Score MMAs K0 .. K1-1 of a block (16 columns each, K1 - K0 even). The tensor pipe takes few instructions ahead,
// so every instruction of the issuing loop shows up in the MMA rate: a loop with a run-time count and the
// descriptor arithmetic per MMA ran at 46 ns per MMA, this one at about 31 (the rate of the MMA itself). Two MMAs
// per iteration rather than the whole sequence unrolled: the fully unrolled issue code made the softmax warps of
// some SMs twice as slow (instruction fetch), the same on every launch.
template <int K0, int K1>
__device__ __forceinline__ void issue_qk(uint32_t dst, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
  static_assert((K1 - K0) % 2 == 0, "two MMAs per iteration");
  uint32_t a = a_tmem + 8u * K0;
  uint64_t b = b_desc + (uint64_t)(16 * K0);
#pragma unroll 1
  for (int kk = K0; kk < K1; kk += 2) {
    mma_bf16_ta(dst, a, b, idesc, kk != 0 ? 1u : 0u);
    mma_bf16_ta(dst, a + 8, b + 16, idesc, 1u);
    a += 16;
    b += 32;
  }
}
__device__ __forceinline__ void mma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
               : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane (the warp reads its 32-lane quarter together)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint4 (&v)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z), "r"(v[1].w),
      "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// One softmax warp's part of the output: its 32 heads, columns c_lo .. c_lo + 127 of the CTA's value half:
// out[h][c] = w0 * O[h][c] (+ w1 * out[h][c], what the CTA of the other key half left there, wherever that head's
// w1 != 0), O read from tensor memory (zero without it). Each thread holds its head's row; 32-column slices go
// through a shared tile (rows 144 bytes apart: conflict-free 16-byte accesses both ways) so that the global reads and
// writes are whole 128-byte row segments.
__device__ __forceinline__ void store_out_rows(uint32_t trow, bool have_o, float w0, float w1, float* tile,
                                               float* rows, int lane, int c_lo) {
  constexpr int TS = 36;  // tile row stride in floats
  const bool merge = __any_sync(0xffffffffu, w1 != 0.f);
  const int col4 = lane & 7;
  for (int c0 = c_lo; c0 < c_lo + DV_HALF / 2; c0 += 32) {
    float o[32];
    if (have_o) {
      tmem_ld16(trow + TMEM_O + c0, *reinterpret_cast<float(*)[16]>(o));
      tmem_ld16(trow + TMEM_O + c0 + 16, *reinterpret_cast<float(*)[16]>(o + 16));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(tile + lane * TS + 4 * q) =
          make_float4(o[4 * q] * w0, o[4 * q + 1] * w0, o[4 * q + 2] * w0, o[4 * q + 3] * w0);
    __syncwarp();
    float4 v[8], o1[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int hl = 4 * r + (lane >> 3);
      v[r] = *reinterpret_cast<const float4*>(tile + hl * TS + 4 * col4);
      if (merge) o1[r] = __ldcg(reinterpret_cast<const float4*>(rows + (size_t)hl * DV + c0 + 4 * col4));
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int hl = 4 * r + (lane >> 3);
      const float w1h = __shfl_sync(0xffffffffu, w1, hl);
      if (merge && w1h != 0.f) {
        v[r].x += w1h * o1[r].x;
        v[r].y += w1h * o1[r].y;
        v[r].z += w1h * o1[r].z;
        v[r].w += w1h * o1[r].w;
      }
      *reinterpret_cast<float4*>(rows + (size_t)hl * DV + c0 + 4 * col4) = v[r];
    }
    __syncwarp();
  }
}

// Address of the row an index names, or nullptr for padding / out-of-range entries (masked keys).
__device__ __forceinline__ const uint8_t* row_of(const MlaArgs& a, int b, int32_t e) {
  if (e >= 0) return e < a.limit ? a.rows + (size_t)b * (size_t)a.req_stride + (size_t)e * ROW_BYTES : nullptr;
  if (a.mode == 0 && e <= -2 && a.resident) {
    const long long r = -2LL - (long long)e;
    return r < a.resident_count ? a.resident + (size_t)r * ROW_BYTES : nullptr;
  }
  return nullptr;
}

__global__ void __launch_bounds__(NTHREADS, 1) hs_mla_decode_kernel(const MlaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // cluster of 2 * nsplit CTAs per request: rank = 2 * split + half; split s takes the s-th run of key blocks,
  // half the score-GEMM columns, and the pair of a split exchanges partial scores
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / (2 * a.nsplit), half = (int)(rank & 1u), split = (int)(rank >> 1);
  const uint32_t peer = rank ^ 1u;
  const int k = a.k, nb_all = (k + KB - 1) / KB, nb_split = (nb_all + a.nsplit - 1) / a.nsplit;
  const int jb = min(nb_all, split * nb_split);  // this split's first block
  const int nb = min(nb_all, jb + nb_split) - jb;  // and its block count (the blocks below are numbered from jb)
  // this CTA's score-GEMM columns: [d0, d0 + 8 * nch)
  const int d0 = half ? DSPLIT : 0, nch = (half ? DQK - DSPLIT : DSPLIT) / 8, grp = (nch + 1) * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t *kfull = bars, *kempty = bars + NSTAGE, *sfull = bars + 2 * NSTAGE, *sempty = sfull + 1,
           *pfull = sempty + 1, *pdone = pfull + NPB, *odone = pdone + NPB, *drain = odone + 1, *xfull = drain + 1,
           *xempty = xfull + 1, *xread = xempty + 1, *tdone = xread + 1, *pmx = tdone + 1, *qready = pmx + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* stage_stop = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
  // [stage][half]: bit i = key half * 32 + i of the stage's block has a row
  uint32_t* kmask = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 8 + 4 * NSTAGE);
  float* pshare = reinterpret_cast<float*>(smem + OFF_PMAX);  // [parity][key half][head]: block maxima, normalisers
  const uint8_t** keyp = reinterpret_cast<const uint8_t**>(smem + OFF_KEY);

  // softmax warps: head quarter q (tensor-memory lanes 32 q .. 32 q + 31), key half kh of every block; thread =
  // head h
  const int q = warp & 3, kh = (warp >> 2) & 1, h = q * 32 + lane;
  // Q is the score GEMM's A operand in tensor memory: lane h holds head h's columns of this CTA, two per 32-bit
  // column. The softmax thread (h, kh) loads half of them (nq 16-byte chunks) now and stores them once the tensor
  // memory is allocated.
  const int nq = nch / 2;
  uint4 qv[MAX_NDIM / 16];
  if (warp < SOFTMAX_WARPS) {
    const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((size_t)b * HEADS + h) * DQK + d0) + kh * nq;
#pragma unroll
    for (int i = 0; i < MAX_NDIM / 16; ++i)
      if (i < nq) qv[i] = __ldg(qrow + i);
  }

  // Loaders: the STAGE_WARPS warps of stage s fill it with blocks s, s + NSTAGE, ... (this CTA's columns of each
  // row). Warp lsub of the stage looks up keys lsub * 32 + lane of the block into the stage's row pointers and
  // validity mask, a named barrier hands them to the other warp, every thread copies its share of the 16-byte
  // chunks, and each warp starts its half of the stage's next rows on their way into L2. Each stage's first block
  // is started here, alongside Q, before anything waits, and lands before the barrier below.
  const bool loader = warp >= LOAD_WARP0 && warp < XCHG_WARP;
  const int ls = (warp - LOAD_WARP0) / STAGE_WARPS, lsub = (warp - LOAD_WARP0) % STAGE_WARPS;
  uint8_t* const lst = smem + OFF_K + ls * STAGE_BYTES;
  // the row of this lane's key of block j (its slot-list entry read from global memory)
  auto lookup = [&](int j) -> const uint8_t* {
    const int i = (jb + j) * KB + lsub * 32 + lane;
    return (lsub < 2 && i < k) ? row_of(a, b, ld_fresh(a.idx + (size_t)b * k + i)) : nullptr;
  };
  // publish a block's rows to the stage (the stage must be free) and to the other warp of the stage
  auto publish = [&](const uint8_t* r) {
    if (lsub < 2) {
      keyp[ls * KB + lsub * 32 + lane] = r;
      const uint32_t m = __ballot_sync(0xffffffffu, r != nullptr);
      if (lane == 0) kmask[ls * 2 + lsub] = m;
    }
    named_sync(1 + ls, STAGE_WARPS * 32);
  };
  auto prefetch_next = [&](int j) {
    // this CTA's part of the rows of the stage's next block starts for L2 while these copies land
    const int i2 = (jb + j + NSTAGE) * KB + lsub * 32 + lane;
    if (lsub < 2 && j + NSTAGE < nb && i2 < k) {
      const uint8_t* r2 = row_of(a, b, ld_fresh(a.idx + (size_t)b * k + i2));
      if (r2) prefetch_l2(r2 + d0 * 2, (uint32_t)nch * 16u);
    }
  };
  auto copy_rows = [&](int) {
    // lane = (row rr of an 8-row group, one of 4 consecutive chunks): a warp's copies fill 512 consecutive bytes
    // of shared memory (the group's slots of 4 chunks), and the two warps of the stage take alternate 4-chunk runs
    const int rr = lane & 7, c0 = lsub * 4 + (lane >> 3);
#pragma unroll 1
    for (int g = 0; g < KB / 8; ++g) {
      const uint8_t* src = keyp[ls * KB + g * 8 + rr];
      uint8_t* dst = lst + g * grp + rr * 16;
      if (src) {
        src += d0 * 2;
        for (int c = c0; c < nch; c += 4 * STAGE_WARPS) cp_async16(dst + c * 128, src + c * 16);
      } else {
        for (int c = c0; c < nch; c += 4 * STAGE_WARPS)
          *reinterpret_cast<uint4*>(dst + c * 128) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_commit();
  };
  if (loader && ls < nb) {
    publish(lookup(ls));
    copy_rows(ls);
  }
  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      bar_init(kfull + i, STAGE_WARPS * 32);
      bar_init(kempty + i, 1);
    }
    bar_init(sfull, 1);
    bar_init(sempty, SOFTMAX_THREADS);
    bar_init(qready, SOFTMAX_THREADS);
    for (int i = 0; i < NPB; ++i) {
      bar_init(pfull + i, SOFTMAX_THREADS);
      bar_init(pdone + i, 1);
    }
    bar_init(odone, 1);
    bar_init(drain, 1);
    bar_init(xfull, 1);                  // one local arrival with the byte count; the peer's async stores complete it
    bar_init(xempty, 1);                 // the peer's exchange warp
    bar_init(xread, SOFTMAX_THREADS);    // this CTA's softmax threads have read the buffer
    bar_init(tdone, SOFTMAX_THREADS);    // every softmax thread has made its last tensor-memory read
    for (int i = 0; i < 4; ++i) bar_init(pmx + i, 64);  // the two softmax warps of a head quarter
    *abort_flag = 0;
    for (int i = 0; i < NSTAGE; ++i) stage_stop[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    bar_arrive_expect(xfull, X_BYTES);  // block 0 of the peer's partial scores is expected in the buffer
  }
  // no key of the second half until its CTA says otherwise (it writes after the first cluster barrier)
  if (tid < HEADS) reinterpret_cast<float2*>(smem + OFF_COMB)[tid] = make_float2(-INFINITY, 0.f);
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tslot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  cp_async_wait_all();
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either touches the other's shared memory
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
  if (warp < SOFTMAX_WARPS) {
#pragma unroll
    for (int c = 0; c < MAX_NDIM / 64; ++c)
      if (4 * c < nq)
        tmem_st16u(trow + TMEM_Q + 4 * kh * nq + 16 * c,
                   *reinterpret_cast<const uint4(*)[4]>(qv + 4 * c));
    tmem_wait_st();
    tc_fence_before();
    bar_arrive(qready);
  }
  // this warp's output rows (32 heads of the CTA's value half) and a shared tile for writing them (the key stages
  // are free by then)
  float* const orows = a.out + ((size_t)b * HEADS + q * 32) * DV + half * DV_HALF;
  float* const otile = reinterpret_cast<float*>(smem + OFF_K) + (warp & 7) * 32 * 36;
  float m_run = -INFINITY, l_run = 0.f;
  bool sm_ok = false;
  // with two key halves, the CTA of split s merges heads 64 s .. 64 s + 63 (head quarters 2 s and 2 s + 1) and
  // hands the other heads to its counterpart
  const bool merges = a.nsplit == 1 || (q >> 1) == split;
  const unsigned lim = a.wait_limit;

  if (loader) {
    // ---- loaders (see above): the first block of each stage has landed; later blocks wait until the value GEMM
    //      of the block NSTAGE earlier has read the stage. Both warps of a stage learn the outcome of the wait at a
    //      named barrier, so they leave the loop together.
    if (ls < nb) {
      bar_arrive(kfull + ls);
      prefetch_next(ls);
    }
    for (int j = ls + NSTAGE; j < nb; j += NSTAGE) {
      // the block's slot-list entries are read while the stage is still in use; only the copy waits for it
      const uint8_t* r = lookup(j);
      if (lsub == 0) {
        const bool ok =
            __all_sync(0xffffffffu, bar_wait(kempty + ls, (unsigned)((j / NSTAGE) - 1) & 1u, abort_flag, lim));
        if (!ok && lane == 0) stage_stop[ls] = 1;
      }
      named_sync(1 + ls, STAGE_WARPS * 32);
      if (stage_stop[ls]) break;
      publish(r);
      copy_rows(j);
      prefetch_next(j);
      cp_async_wait_all();
      fence_proxy_async();
      bar_arrive(kfull + ls);
    }
    cp_async_wait_all();
  } else if (warp == XCHG_WARP) {
    // ---- exchange warp: once this CTA's softmax threads have read block j from the exchange buffer, it expects
    //      block j + 1 there and lets the peer send it. Its acquire (wait) and release (remote arrive) carry the
    //      softmax threads' reads before the peer's next stores, and keep that release off their critical path.
    if (lane == 0) {
      for (int j = 0; j < nb; ++j) {
        if (!bar_wait(xread, (unsigned)j & 1u, abort_flag, lim)) break;
        if (j + 1 < nb) {
          bar_arrive_expect(xfull, X_BYTES);
          bar_arrive_peer(peer_addr(xempty, peer));
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ---- one thread issues the tensor-core work: partial scores of block j over this CTA's columns, and the
    //      value GEMM of block j - 1 for this CTA's value half
    if (lane == 0) {
      const uint32_t k0 = su32(smem + OFF_K), p0 = su32(smem + OFF_P), tq = tmem + TMEM_Q;
      constexpr uint32_t ID_QK = idesc_bf16(128, KB, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16(128, DV_HALF, 0, 1);
      // Descriptors are built once; an operand 256 bytes further along is the same descriptor plus 16 in its start
      // field (shared-memory addresses stay below 256 KB, so the 14-bit field never carries).
      const uint64_t dk = sdesc(k0, 128, grp), dp = sdesc(p0, 128, P_GROUP),
                     dv = sdesc(k0, grp, 128);
      // test hook: wait on a barrier that nothing completes (drain: its only arrival is the commit below), before
      // anything is issued, so that the wait runs out with no tensor-core work or copy of this CTA in flight
      bool ok = !a.stall || bar_wait(drain, 0, abort_flag, lim);
      ok = ok && bar_wait(qready, 0, abort_flag, lim);
      // The value GEMM of block j-1 goes in as soon as its P is ready: pfull is polled halfway through the score
      // GEMM of block j (the tensor pipe runs in issue order), so the key stage of block j-1 is released without
      // waiting for all of block j's scores.
      auto issue_pv = [&](int jp) {
        const int s = jp % NSTAGE, pb = jp % NPB;
        tc_fence_after();
        // P (K-major: keys are K) times this CTA's value half of the key rows, its first 256 columns (MN-major:
        // the value columns are N), 16 keys (two 8-key groups) per MMA
        const uint64_t da = dp + (uint64_t)((pb * P_BYTES) >> 4), db = dv + (uint64_t)((s * STAGE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk)
          mma_bf16(tmem + TMEM_O, da + (uint64_t)(16 * kk), db + (uint64_t)(kk * ((2 * grp) >> 4)), ID_PV,
                   (jp > 0 || kk > 0) ? 1u : 0u);
        mma_commit(kempty + s);
        mma_commit(pdone + pb);
        if (jp == nb - 1) mma_commit(odone);
      };
      for (int j = 0; j <= nb && ok; ++j) {
        bool pv_pending = j >= 1;
        const int jp = j - 1;
        if (j < nb) {
          const int s = j % NSTAGE;
          ok = bar_wait(kfull + s, (unsigned)(j / NSTAGE) & 1u, abort_flag, lim);
          // one score buffer: block j's scores go in once every softmax thread has read block j - 1's
          if (ok && j >= 1) ok = bar_wait(sempty, (unsigned)(j - 1) & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dkb = dk + (uint64_t)((s * STAGE_BYTES) >> 4);
          const uint32_t dst = tmem + TMEM_S;
          constexpr int NK0 = DSPLIT / 16, NK1 = (DQK - DSPLIT) / 16;  // score MMAs of CTA 0 and CTA 1
          if (half == 0)
            issue_qk<0, NK0 / 2>(dst, tq, dkb, ID_QK);
          else
            issue_qk<0, NK1 / 2>(dst, tq, dkb, ID_QK);
          if (pv_pending && bar_poll(pfull + jp % NPB, (unsigned)(jp / NPB) & 1u)) {
            issue_pv(jp);
            pv_pending = false;
          }
          if (half == 0)
            issue_qk<NK0 / 2, NK0>(dst, tq, dkb, ID_QK);
          else
            issue_qk<NK1 / 2, NK1>(dst, tq, dkb, ID_QK);
          mma_commit(sfull);
        }
        if (pv_pending) {
          ok = bar_wait(pfull + jp % NPB, (unsigned)(jp / NPB) & 1u, abort_flag, lim);
          if (!ok) break;
          issue_pv(jp);
        }
      }
      // every issued MMA has finished before the tensor memory is freed
      mma_commit(drain);
      bool drained = false;
      for (unsigned it = 0; it < WAIT_LIMIT && !(drained = bar_test(drain, 0)); ++it) {
      }
      if (!drained) *abort_flag = 1;
    }
    __syncwarp();
  } else {
    // ---- softmax: thread h of warp w holds head h = TMEM lane h for the keys of its half (kh) of every block. The
    //      partial scores of a block go to the peer, whose partial scores come back; both CTAs then hold S = own +
    //      peer (the same value in both, addition commutes) and run the same softmax, so their P, running max and
    //      normaliser agree bit for bit. The two threads of a head (warps q and q + 4) agree on the block maximum
    //      through shared memory and a per-quarter mbarrier; each keeps the sum of its own weights.
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int s = j % NSTAGE;
      ok = __all_sync(0xffffffffu, ok && bar_wait(sfull, (unsigned)j & 1u, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      float sv[KH];
#pragma unroll
      for (int c = 0; c < KH; c += 16)
        tmem_ld16(trow + TMEM_S + kh * KH + c, *reinterpret_cast<float(*)[16]>(sv + c));
      tc_fence_before();
      bar_arrive(sempty);
      // the peer's exchange buffer is free once the peer has read block j - 1 from it
      if (j >= 1) {
        ok = __all_sync(0xffffffffu, bar_wait_cluster(xempty, (unsigned)(j - 1) & 1u, abort_flag, lim));
        if (!ok) break;
      }
      // exchange buffer layout: float4 group g (scores 4g..4g+3 of the block) of head h at (g * HEADS + h) * 16; the
      // stores complete the transaction bytes of the peer's xfull barrier, which the peer set up in advance
      const uint8_t* xmine = smem + OFF_X;
      const uint32_t xpeer = peer_addr(xmine + h * 16, peer), xfull_peer = peer_addr(xfull, peer);
#pragma unroll
      for (int g = 0; g < KH / 4; ++g)
        st_peer_async_v4(xpeer + (kh * (KH / 4) + g) * HEADS * 16, sv[4 * g], sv[4 * g + 1], sv[4 * g + 2],
                         sv[4 * g + 3], xfull_peer);
      ok = __all_sync(0xffffffffu, bar_wait_cluster(xfull, (unsigned)j & 1u, abort_flag, lim));
      if (!ok) break;
#pragma unroll
      for (int g = 0; g < KH / 4; ++g) {
        const float4 o = *reinterpret_cast<const float4*>(xmine + ((kh * (KH / 4) + g) * HEADS + h) * 16);
        sv[4 * g] += o.x;
        sv[4 * g + 1] += o.y;
        sv[4 * g + 2] += o.z;
        sv[4 * g + 3] += o.w;
      }
      bar_arrive(xread);  // the exchange warp hands the buffer back to the peer
      // which keys of the block have a row (written by the loaders before they signalled the stage full)
      ok = __all_sync(0xffffffffu, bar_wait(kfull + s, (unsigned)(j / NSTAGE) & 1u, abort_flag, lim));
      if (!ok) break;
      const uint32_t vm = kmask[s * 2 + kh];
      float x[KH];
      float mb = -INFINITY;
#pragma unroll
      for (int i = 0; i < KH; ++i) {
        x[i] = (vm >> i) & 1u ? sv[i] * a.scale_log2 : -INFINITY;
        mb = fmaxf(mb, x[i]);
      }
      // the block maximum over both halves of the keys
      float* const share = pshare + (j & 1) * 2 * HEADS;
      share[kh * HEADS + h] = mb;
      bar_arrive(pmx + q);
      ok = __all_sync(0xffffffffu, bar_wait(pmx + q, (unsigned)j & 1u, abort_flag, lim));
      if (!ok) break;
      mb = fmaxf(mb, share[(kh ^ 1) * HEADS + h]);
      float m_new = m_run;
      if (mb > -INFINITY && (m_run == -INFINITY || mb > m_run + 8.f)) m_new = mb;
      const bool resc = m_new != m_run && m_run != -INFINITY;
      if (__any_sync(0xffffffffu, resc)) {
        // O holds blocks 0 .. j-1 once the value GEMM of block j-1 has finished; scale this thread's half of its
        // head's row (both threads of the head take the same decision)
        ok = __all_sync(0xffffffffu,
                        bar_wait(pdone + ((j - 1) % NPB), (unsigned)((j - 1) / NPB) & 1u, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        const float f = resc ? ex2_approx(m_run - m_new) : 1.f;
        for (int c = kh * (DV_HALF / 2); c < (kh + 1) * (DV_HALF / 2); c += 16) {
          float o[16];
          tmem_ld16(trow + TMEM_O + c, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= f;
          tmem_st16(trow + TMEM_O + c, o);
        }
        tmem_wait_st();
        l_run *= f;
      }
      m_run = m_new;
      uint32_t pk[KH / 2];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < KH / 2; ++i) {
        // both weights rounded to bf16 by one conversion (key 2i in the low half)
        const __nv_bfloat162 p2 =
            __floats2bfloat162_rn(x[2 * i] == -INFINITY ? 0.f : ex2_approx(x[2 * i] - m_run),
                                  x[2 * i + 1] == -INFINITY ? 0.f : ex2_approx(x[2 * i + 1] - m_run));
        const float2 pf = __bfloat1622float2(p2);
        psum += pf.x + pf.y;
        pk[i] = *reinterpret_cast<const uint32_t*>(&p2);
      }
      l_run += psum;
      // P buffer pb is free once the value GEMM of block j - NPB has read it
      const int pb = j % NPB;
      if (j >= NPB) {
        ok = __all_sync(0xffffffffu, bar_wait(pdone + pb, (unsigned)((j - NPB) / NPB) & 1u, abort_flag, lim));
        if (!ok) break;
      }
      uint8_t* prow = smem + OFF_P + pb * P_BYTES + (h >> 3) * P_GROUP + (h & 7) * 16;
#pragma unroll
      for (int c = 0; c < KH / 8; ++c)
        *reinterpret_cast<uint4*>(prow + (kh * (KH / 8) + c) * 128) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async();
      tc_fence_before();
      bar_arrive(pfull + pb);
    }
    if (ok && nb > 0) ok = __all_sync(0xffffffffu, bar_wait(odone, 0, abort_flag, lim));
    if (ok) {
      // the head's normaliser: the two threads' sums (the running max is already common)
      float* const share = pshare + (nb & 1) * 2 * HEADS;
      share[kh * HEADS + h] = l_run;
      bar_arrive(pmx + q);
      ok = __all_sync(0xffffffffu, bar_wait(pmx + q, (unsigned)nb & 1u, abort_flag, lim));
      if (ok) l_run += share[(kh ^ 1) * HEADS + h];
    }
    sm_ok = ok;
    if (ok && !merges) {
      // heads the other key half merges: this half's normalised output goes to `out` (this CTA's columns), and
      // (m, l) to the CTA of the other half with the same columns
      tc_fence_after();
      store_out_rows(trow, nb > 0, l_run > 0.f ? 1.f / l_run : 0.f, 0.f, otile, orows, lane, kh * (DV_HALF / 2));
      if (kh == 0) st_peer_v2(peer_addr(smem + OFF_COMB + h * 8, rank ^ 2u), m_run, l_run);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peers no longer touch this CTA's shared memory, and the second half's outputs are written
  if (warp < SOFTMAX_WARPS && sm_ok && merges) {
    // merge with the other key half (none: m1 = -inf, l1 = 0): with M = max(m0, m1) and c_s = 2^(m_s - M),
    // out = (c0 O0 + c1 l1 out1) / (c0 l0 + c1 l1), lse = ln 2 * (M + log2(c0 l0 + c1 l1))
    tc_fence_after();
    const float2 ml1 = *reinterpret_cast<const float2*>(smem + OFF_COMB + h * 8);
    const float m1 = a.nsplit > 1 ? ml1.x : -INFINITY, l1 = a.nsplit > 1 ? ml1.y : 0.f;
    const float mx = fmaxf(m_run, m1);
    const float c0 = l_run > 0.f ? ex2_approx(m_run - mx) : 0.f, c1 = l1 > 0.f ? ex2_approx(m1 - mx) : 0.f;
    const float lsum = c0 * l_run + c1 * l1;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    store_out_rows(trow, nb > 0, c0 * inv, c1 * l1 * inv, otile, orows, lane, kh * (DV_HALF / 2));
    if (half == 0 && kh == 0)
      a.lse[(size_t)b * HEADS + h] = lsum > 0.f ? (mx + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
  }
  // The tensor memory is freed once every softmax thread has arrived on tdone after its last read of it (a
  // per-thread arrival count: a CTA-wide bar.sync here was seen to let the other warps through while two warps
  // were still in the merge, so it does not order the free after those reads). The wait is bounded but does not
  // stop at the abort flag: aborted threads skip their reads and arrive at once.
  if (warp < SOFTMAX_WARPS) {
    tc_fence_before();
    bar_arrive(tdone);
  }
  if (warp == MMA_WARP) {
    if (lane == 0) {
      bool done = false;
      for (unsigned it = 0; it < WAIT_LIMIT && !(done = bar_test(tdone, 0)); ++it) {
      }
      if (!done) *abort_flag = 1;  // a softmax thread never arrived: report it like any other wait that ran out
      if (*abort_flag) atomicOr(a.err, HS_DEVERR_TIMEOUT);
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// How many clusters of four CTAs (a request's two key halves) the current device holds at once, cached per device.
int four_cta_clusters_resident() {
  static std::atomic<int> cache[64];  // 0: not yet asked, else the count + 1
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  const int c = cache[dev].load(std::memory_order_relaxed);
  if (c) return c - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4, 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 4;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, hs_mla_decode_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev].store(n + 1, std::memory_order_relaxed);
  return n;
}

// Failure-detection test settings (hs_debug_attention_waits): the role-wait limit and the stall hook.
std::atomic<unsigned> g_wait_limit{WAIT_LIMIT};
std::atomic<int> g_stall{0};

int launch_mla(hs_pool* p, int32_t batch, MlaArgs a, cudaStream_t s) {
  if (cudaFuncSetAttribute(hs_mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_UNSUPPORTED;
  }
  // Split each request's keys in two (a cluster of four CTAs) when every request's cluster fits on the device at
  // once; the per-block chain of dependent steps, not a bandwidth, bounds a CTA pair, so twice the SMs take half
  // the blocks each.
  a.nsplit = four_cta_clusters_resident() >= batch ? 2 : 1;
  a.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  a.stall = g_stall.load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * a.nsplit * batch), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // the CTAs of a request
  attr[1].val.clusterDim.x = (unsigned)(2 * a.nsplit);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  (void)p;
  return cudaLaunchKernelEx(&cfg, hs_mla_decode_kernel, a) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

bool common_args_ok(const hs_pool* p, int32_t layer, int32_t batch, const void* q, const int32_t* idx, int32_t k,
                    const float* out, const float* lse) {
  if (!p || layer < 0 || layer >= p->d.layers || batch < 0 || batch > p->d.max_batch || k < 0) return false;
  if (batch == 0 || k == 0) return true;
  return q && idx && out && lse && !(reinterpret_cast<uintptr_t>(q) & 15) && !(reinterpret_cast<uintptr_t>(out) & 15);
}

}  // namespace

extern "C" int hs_mla_decode(hs_pool* pool, int32_t layer, int32_t batch, const void* q, const int32_t* out_slots,
                             int32_t k, const void* resident_rows, int64_t resident_count, float sm_scale, float* out,
                             float* lse, hs_stream_t stream) {
  if (!common_args_ok(pool, layer, batch, q, out_slots, k, out, lse) || resident_count < 0 ||
      (resident_rows && (reinterpret_cast<uintptr_t>(resident_rows) & 15)))
    return HS_ERR_INVALID_ARG;
  if (pool->d.row_bytes != ROW_BYTES) return HS_ERR_UNSUPPORTED;
  if (batch == 0 || k == 0) return HS_OK;
  const size_t hrl = (size_t)pool->d.slots * ROW_BYTES;
  MlaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint16_t*>(q);
  a.idx = out_slots;
  a.k = k;
  a.mode = 0;
  a.rows = static_cast<const uint8_t*>(pool->d.hot_buf) + (size_t)layer * (size_t)pool->d.max_batch * hrl;
  a.req_stride = (int64_t)hrl;
  a.limit = pool->d.slots;
  a.resident = static_cast<const uint8_t*>(resident_rows);
  a.resident_count = resident_rows ? resident_count : 0;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.err = pool->err;
  return launch_mla(pool, batch, a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int hs_mla_decode_history(hs_pool* pool, int32_t layer, int32_t batch, const void* q,
                                     const int32_t* topk_idx, int32_t k, float sm_scale, float* out, float* lse,
                                     hs_stream_t stream) {
  if (!common_args_ok(pool, layer, batch, q, topk_idx, k, out, lse)) return HS_ERR_INVALID_ARG;
  if (pool->d.row_bytes != ROW_BYTES) return HS_ERR_UNSUPPORTED;
  if (batch == 0 || k == 0) return HS_OK;
  MlaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint16_t*>(q);
  a.idx = topk_idx;
  a.k = k;
  a.mode = 1;
  a.rows = pool->src + (size_t)layer * (size_t)pool->d.host_layer_stride;
  a.req_stride = pool->d.host_req_stride ? pool->d.host_req_stride : (int64_t)pool->d.ctx * ROW_BYTES;
  a.limit = pool->d.ctx;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.err = pool->err;
  return launch_mla(pool, batch, a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int hs_debug_attention(uint32_t wait_limit, int32_t stall, int32_t* split_max_batch) {
  g_wait_limit.store(wait_limit ? wait_limit : WAIT_LIMIT, std::memory_order_relaxed);
  g_stall.store(stall ? 1 : 0, std::memory_order_relaxed);
  if (split_max_batch) *split_max_batch = four_cta_clusters_resident();
  return HS_OK;
}
