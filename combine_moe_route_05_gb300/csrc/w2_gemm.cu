// Router-score absorption fused into the W2 grouped GEMM, on the fifth-
// generation tensor cores (tcgen05 MMA on a CTA pair, accumulators in tensor
// memory, TMA operand loads).
//
// What it computes ([Titan-absorb] "Implementation": the W2 input is scaled by
// the routed score in float32 and restored to its dtype before the grouped
// GEMM; the pages' "FusedMOE" section names an SM100+ fused MoE backend as the
// direction): for every receive row r of expert e's segment,
//   hs[r,i] = round_bf16(h[r,i] * recv_w[r])
//   y[r,n]  = round_bf16(sum_i hs[r,i] * W2[e][n,i])      (fp32 accumulation)
// with W2 stored [E][H][I].  The scaling is the GEMM's prologue: the scaled
// rows never reach HBM.  A pad row of a padded layout gets y = 0.
//
// Persistent clusters of two CTAs (a CTA pair) walk 256 x 384 output tiles:
// each CTA owns 128 rows (adjacent 128-row m-tiles of one expert; each
// expert's segment is cut into 128-row tiles, the last one ragged) and half
// of the tile's 384 W2 columns in shared memory.  Two MMA instructions of the
// pair per K step, issued by the even CTA, multiply all 256 rows by the
// tile's two 192-column halves; each CTA keeps its 128 x 384 accumulator in
// its own tensor memory (384 of its 512 columns; the other 128 hold four
// scaled-h stages).  Per CTA and 64-wide K slice, shared memory carries 16 KB
// of h and 24 KB of W2 landed by TMA, 16 KB of h read by the prologue and
// 24 KB of W2 read by the tensor cores, 80 KB for 768 cycles of MMAs (a
// 256-column tile moved 64 KB for 512).  The h slice of a row block is
// scaled once per 384 output columns.  Where H is not a multiple of 384 the
// last tile of a row of tiles computes its full width and stores only the
// columns inside H (narrower MMAs for it measured slower).
//
// Warp roles, in both CTAs:
//   warp 2      TMA: h slices [128 x 64] into a 4-stage ring (128-byte
//               swizzle), freed once the prologue has consumed them (after
//               its tensor-memory store: the refill must not overtake the
//               prologue's shared-memory loads);
//   warp 0      TMA: this CTA's part of each W2 slice, [96 x 64] for each
//               of the two column halves, into a 4-stage ring.  The copies
//               of BOTH CTAs complete on the even CTA's `full` barrier of the
//               stage (the pair form of the bulk tensor copy lets the barrier
//               sit in the peer CTA), and the even CTA's producer announces
//               the bytes of both CTAs;
//   warps 3-6   prologue: read an h slice (one row per thread, one warp per
//               tensor-memory lane quarter), scale it by the row's score
//               (fp32 product, bf16 round-to-nearest-even), store it into the
//               32-column A stage in tensor memory that pairs with the W2
//               stage of the same index; the four warps meet at a named
//               barrier, and one thread arrives on the even CTA's `full`
//               barrier for the CTA (two remote arrivals per slice, not one
//               per warp);
//   warp 1      tensor memory (allocated by the pair together: a 384-column
//               accumulator + four A stages); in the even CTA one thread
//               waits on `full` (both CTAs' W2 parts and both CTAs' A
//               stages), issues the pair's MMAs (two halves of
//               four K=16 steps per slice; a tile's first MMAs into a half
//               wait until the epilogue has read that half) and commits, once
//               to each CTA's `empty` barrier of the stage and, per tile, to
//               each CTA's `acc_full`;
//   warps 7-14  epilogue: per column half, accumulator -> registers (two
//               warps per lane quarter, 96 columns each), the half handed
//               back (an arrival on the even CTA's `acc_empty` of the half),
//               then bf16 rows to HBM while the next tile's MMAs run.
// Every wait is bounded; a wait that gives up raises MOE_DEVERR_TIMEOUT and
// the CTA winds down (copies in flight are waited for, tensor memory freed).
// No load is multicast: each CTA loads its own rows of h and its own half of
// W2.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kBM = 128;          // rows per CTA: the accumulator's tensor-memory lanes
constexpr int kMmaN = 192;            // columns of one MMA instruction of the pair
constexpr int kHalves = 2;            // MMAs per K step: the tile's two column halves
constexpr int kBN = kHalves * kMmaN;  // output columns per tile
constexpr int kSubRows = kMmaN / 2;   // W2 rows one CTA holds for one MMA half
constexpr int kBNHalf = kBN / 2;      // W2 rows held by one CTA
constexpr int kHMultiple = 256;       // the entry point's contract: H a multiple of 256
constexpr int kBK = 64;           // contraction per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;        // contraction per MMA instruction (16-bit operands)
constexpr int kStagesA = 4;       // h slices in shared memory
// W2 half-slices in shared memory and scaled h slices in tensor memory share
// one ring index: one barrier says "both operands of slice j are in place in
// both CTAs", one commit per CTA frees both
constexpr int kStages = 4;
constexpr int kPrologueWarps = 4;  // one per lane quarter, the whole K range of a slice
constexpr int kEpilogueWarps = 8;  // two per lane quarter, half the columns each
constexpr int kFirstPrologueWarp = 3;
constexpr int kFirstEpilogueWarp = kFirstPrologueWarp + kPrologueWarps;
constexpr int kThreads = 32 * (kFirstEpilogueWarp + kEpilogueWarps);
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr uint32_t kSubBytes = kSubRows * kBK * 2;  // one MMA half's W2 rows of a CTA
constexpr uint32_t kBBytes = kHalves * kSubBytes;
static_assert(kSubBytes % 1024 == 0, "W2 sub-tiles start on 1024-byte swizzle boundaries");
constexpr uint32_t kAccCols = kBN;    // fp32 accumulator: a column per output column
constexpr uint32_t kACols = kBK / 2;  // a scaled h slice: two bf16 per 32-bit column
constexpr uint32_t kTmemCols = 512;   // accumulator + kStages A stages (power of 2)
static_assert(kAccCols + kStages * kACols <= kTmemCols, "tensor memory budget");
constexpr size_t kBarrierBytes = 512;
static_assert(8 * (2 * kStagesA + 2 * kStages + 1 + kHalves) + 16 <= kBarrierBytes, "barrier area");
// operand rings, barriers and the tables of at most MOE_MAX_EXPERTS experts
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStagesA * kABytes + kStages * kBBytes +
                              kBarrierBytes + sizeof(int32_t) * (3 * MOE_MAX_EXPERTS + 2);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kSmemBytes < (1u << 18), "descriptor start addresses fit 14 bits of 16 bytes");

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A
// and B bf16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3
// in bits 17-22, M >> 4 in bits 24-28; M = 256 rows over the CTA pair.
constexpr uint32_t kIdescNoN = (1u << 4) | (1u << 7) | (1u << 10) |
                               (static_cast<uint32_t>((2 * kBM) >> 4) << 24);
__host__ __device__ constexpr uint32_t idesc_for(int n) {
  return kIdescNoN | (static_cast<uint32_t>(n >> 3) << 17);
}


struct W2Args {
  const float* recv_w;
  const int32_t* off_e;
  const int32_t* cnt_e;
  __nv_bfloat16* y;
  uint32_t* flags;
  unsigned long long wait_ns;  // limit of every mbarrier wait
  int rows;                    // receive rows of h and y (T*K plus the pads)
  int E, I, H;
  int n_tiles;  // ceil(H / kBN): the last tile's columns past H are not stored
};

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzle layout (rows of 128 bytes, 8-row groups 1024 bytes apart): start
// address >> 4 in bits 0-13, leading offset 16 B (unused by this layout) in
// bits 16-29, stride offset 1024 B >> 4 in bits 32-45, descriptor version 1 in
// bits 46-47, base offset 0 (tiles are 1024-byte aligned), swizzle mode 2
// (128-byte) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity; false after limit_ns.
// Every wait and arrival here has the default semantics (acquire / release at
// CTA scope), also across the pair: what crosses between the CTAs is tensor
// memory (ordered by the tcgen05 fences around the barrier) and the bulk
// copies (complete_tx makes them visible to the thread that observes the
// phase).  Cluster-scope releases cost about 0.6 us each on this part, which
// at one per slice and warp made the pair slower than a single CTA.
// The test suspends the thread until the phase completes or about
// kSuspendNs have passed, so that waiting warps (an epilogue waits a whole
// tile) do not spend the issue slots the prologue needs.
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool phase_done(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity,
                                           unsigned long long limit_ns) {
  if (phase_done(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (phase_done(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive on a barrier of either CTA of the pair (`cluster_bar`, a cluster
// shared-memory address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Tensor copy into this CTA's shared memory, completing on a barrier of this
// CTA.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Tensor copy into this CTA's shared memory, completing on a barrier of
// either CTA of the pair (`cluster_bar`, a cluster shared-memory address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}

// AND of `p` over the nthreads threads (whole warps) that meet at named
// barrier `id`; every one of them must reach it.
__device__ __forceinline__ bool bar_and(bool p, int id, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T over the CTA pair (issued by the even
// CTA): A rows 0-127 from this CTA's tensor memory and 128-255 from the
// peer's, B columns 0-127 from this CTA's shared memory and 128-255 from the
// peer's (same addresses); each CTA's tensor memory receives its 128 rows.
// A in tensor memory: lane = row, 32-bit column j = bf16 elements 2j, 2j+1.
__device__ __forceinline__ void umma_pair(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc,
                                          uint32_t accumulate, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %3, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b_desc), "r"(accumulate), "r"(idesc)
      : "memory");
}

// Arrive on the barrier at cluster shared-memory address `cluster_bar` (in
// either CTA of the pair) once every MMA this thread issued so far has
// completed.
__device__ __forceinline__ void umma_commit_to(uint32_t cluster_bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          cluster_bar)
      : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.  The
// store reads its source registers asynchronously, so the store and its wait
// are one asm statement: the registers stay reserved until the wait returns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.  The
// load and its wait are one asm statement: the load is asynchronous, and the
// registers are defined only once the wait has returned, so no use of them
// may be scheduled in between.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Shared-memory tables of one CTA: the layout's expert segments and, per
// expert, the index of its first pair of 128-row m-tiles (tile_first[E] = all
// pairs).
struct Tables {
  int32_t* tile_first;  // [E + 1]
  int32_t* off;         // [E + 1]
  int32_t* cnt;         // [E]
};

struct Tile {
  int expert, row0, nt;
  int seg_end;   // end of the expert's segment (pads included)
  int real_end;  // end of the expert's real rows
};

// Pair tile `tile` (n-tile fastest) -> expert and this CTA's rows: the last
// expert whose first pair is <= the tile's pair (an empty expert shares its
// first pair with the next expert and is never the last such one).  CTA
// `rank` takes m-tile 2 * pair + rank of the expert; past the expert's last
// m-tile it has no rows (row0 >= seg_end) but still holds its W2 half.
__device__ __forceinline__ Tile decode_tile(const Tables& tb, int E, int n_tiles, int tile,
                                            int rank) {
  const int mt = tile / n_tiles;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.tile_first[mid] <= mt)
      lo = mid;
    else
      hi = mid - 1;
  }
  Tile t;
  t.expert = lo;
  t.nt = tile - mt * n_tiles;
  t.row0 = tb.off[lo] + (2 * (mt - tb.tile_first[lo]) + rank) * kBM;
  t.seg_end = tb.off[lo + 1];
  t.real_end = tb.off[lo] + tb.cnt[lo];
  return t;
}

// Persistent: pair p takes pair tiles p, p + npairs, ... in every role of
// both CTAs, so all roles walk the same sequence of (tile, K slice) jobs;
// each ring runs on across tiles.
__global__ void __launch_bounds__(kThreads, 1)
    w2_absorbed_kernel(const __grid_constant__ CUtensorMap tm_h,
                       const __grid_constant__ CUtensorMap tm_w2, W2Args a) {
  extern __shared__ uint8_t smem_raw[];
  // operand tiles start on 1024-byte shared-memory boundaries (the swizzle
  // pattern repeats every 8 rows of 128 bytes); the offsets are the same in
  // both CTAs, as the pair's MMA requires
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                       // [kStagesA][kBM x kBK] bf16, swizzled
  uint8_t* sB = smem + kStagesA * kABytes;  // [kStages][kHalves][kSubRows x kBK] bf16, swizzled
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
  uint64_t* full_a = bars;               // [kStagesA] h slice landed
  uint64_t* free_a = full_a + kStagesA;  // [kStagesA] h slice consumed by the prologue
  uint64_t* full = free_a + kStagesA;    // [kStages] even CTA: both W2 halves, all A stores
  uint64_t* empty = full + kStages;      // [kStages] the pair's MMAs done with the stage
  uint64_t* acc_full = empty + kStages;  // accumulator complete
  uint64_t* acc_empty = acc_full + 1;    // [kHalves] even CTA: that column half drained in both CTAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + kHalves);
  Tables tb;
  tb.tile_first = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(bars) + kBarrierBytes);
  tb.off = tb.tile_first + (a.E + 1);
  tb.cnt = tb.off + (a.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (a.I + kBK - 1) / kBK;
  const int rank = static_cast<int>(cluster_rank());
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  // the segments, checked: 0 <= off[e] <= off[e] + cnt[e] <= off[e+1] <=
  // rows; a layout that breaks this (corrupted or not this handle's) raises
  // MOE_DEVERR_BAD_LAYOUT and the kernel computes nothing (both CTAs of a
  // pair read the same layout and decide alike)
  int bad = 0;
  for (int e = threadIdx.x; e <= a.E; e += kThreads) {
    const int lo = a.off_e[e];
    tb.off[e] = lo;
    if (e < a.E) {
      const int c = a.cnt_e[e], hi = a.off_e[e + 1];
      tb.cnt[e] = c;
      bad |= lo < 0 || c < 0 || c > hi - lo || hi > a.rows;
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && rank == 0) raise_flag(a.flags, MOE_DEVERR_BAD_LAYOUT);
    for (int e = threadIdx.x; e <= a.E; e += kThreads) {
      tb.off[e] = 0;
      if (e < a.E) tb.cnt[e] = 0;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the per-expert counts of m-tile pairs
    int running = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      const int tiles = e < a.E ? ((tb.off[e + 1] - tb.off[e] + kBM - 1) / kBM + 1) / 2 : 0;
      int incl = tiles;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      if (e < a.E) tb.tile_first[e] = running + incl - tiles;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      tb.tile_first[a.E] = running;
      for (int s = 0; s < kStagesA; ++s) {
        mbar_init(&full_a[s], 1);
        mbar_init(&free_a[s], 1);  // one arrival for the CTA's prologue warps
      }
      for (int s = 0; s < kStages; ++s) {
        // even CTA: its W2 producer's arrival (with both halves' bytes) and
        // the prologue warps of both CTAs; the odd CTA's is unused
        mbar_init(&full[s], 1 + 2);  // the W2 producer's arrival, one per CTA's prologue
        mbar_init(&empty[s], 1);  // the pair's commit
      }
      mbar_init(acc_full, 1);                    // the pair's commit
      for (int j = 0; j < kHalves; ++j)
        mbar_init(&acc_empty[j], 2 * kEpilogueWarps);  // epilogue warps of both CTAs
      fence_mbar_init();
    }
  } else if (warp == 1) {
    // the pair allocates together: one warp of each CTA
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
  }
  tc_fence_before();
  // the peer's barriers must be initialised before its arrivals, copies and
  // commits can reach them
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;         // accumulator: columns [0, 256)
  const uint32_t tmem_a = tmem + kAccCols;  // A stages: 32 columns each
  const int total = tb.tile_first[a.E] * a.n_tiles;
  const int my_tiles = pair < total ? (total - pair + npairs - 1) / npairs : 0;

  bool ok = true;
  if (warp == 0 || warp == 2) {
    // TMA producers: warp 0 this CTA's halves of the W2 slices, warp 2 the h
    // slices
    if (lane == 0) {
      const bool is_b = warp == 0;
      const int stages = is_b ? kStages : kStagesA;
      int it = 0;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        const Tile t = decode_tile(tb, a.E, a.n_tiles, tile, rank);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1u;
          if (is_b) {
            // the stage is free in both CTAs once the pair's MMAs that read
            // it have completed (a commit reaches each CTA's `empty`)
            if (it >= stages && !wait_phase(&empty[s], ph ^ 1u, a.wait_ns)) {
              ok = false;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kBBytes);
            // MMA half j takes W2 rows j kMmaN .. j kMmaN + kMmaN - 1 of the
            // tile, the even CTA the first kSubRows of them.  In a ragged last
            // tile the columns past H are not stored, so a box wholly past the
            // expert's rows reads the expert's own last rows again (in L2)
            // instead of the next expert's from HBM
            const int row_end = (t.expert + 1) * a.H;
#pragma unroll
            for (int j = 0; j < kHalves; ++j) {
              const int row = t.expert * a.H + t.nt * kBN + j * kMmaN + rank * kSubRows;
              tma_load_2d_pair(sB + s * kBBytes + j * kSubBytes, &tm_w2, kb * kBK,
                               row < row_end ? row : row_end - kSubRows,
                               cluster_addr(&full[s], 0));
            }
          } else {
            if (it >= stages && !wait_phase(&free_a[s], ph ^ 1u, a.wait_ns)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_a[s], kABytes);
            tma_load_2d(sA + s * kABytes, &tm_h, kb * kBK, t.row0, &full_a[s]);
          }
        }
      }
      // the last copies must have landed before the CTA may exit: for h, its
      // own barrier says so; for W2, the pair's last commits on this CTA's
      // stages (the MMAs that read a stage ran after its copies landed)
      for (int j = it - stages < 0 ? 0 : it - stages; j < it; ++j) {
        if (is_b) {
          if (!wait_phase(&empty[j % stages], (j / stages) & 1u, a.wait_ns)) ok = false;
        } else if (!wait_phase(&full_a[j % stages], (j / stages) & 1u, a.wait_ns)) {
          ok = false;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int it = 0, n = 0;
      const uint32_t acc_full_peer = cluster_addr(acc_full, 1);
      // the stages' `empty` barriers are 8 bytes apart in both CTAs
      const uint32_t empty_own = smem_addr(empty), empty_peer = cluster_addr(empty, 1);
      for (int tile = pair; tile < total && ok; tile += npairs, ++n) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (!wait_phase(&full[s], (it / kStages) & 1u, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the descriptor's start-address field is the address >> 4 (14 bits:
          // shared memory ends below 256 KB), so the other MMAs of the slice
          // add their byte offset >> 4 to the stage's descriptor
          const uint64_t d0 = sw128_desc(smem_addr(sB + s * kBBytes));
#pragma unroll
          for (int j = 0; j < kHalves; ++j) {
            // a tile's first MMAs into a column half wait until the epilogue
            // of both CTAs has read the previous tile's values there
            if (kb == 0 && n >= 1) {
              if (!wait_phase(&acc_empty[j], (n - 1) & 1u, a.wait_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              umma_pair(tmem + j * kMmaN, tmem_a + s * kACols + k * (kUmmaK / 2),
                        d0 + ((j * kSubBytes + k * kUmmaK * 2) >> 4), (kb | k) != 0,
                        idesc_for(kMmaN));
          }
          if (!ok) break;
          // frees the stage in both CTAs
          umma_commit_to(empty_own + 8 * s);
          umma_commit_to(empty_peer + 8 * s);
        }
        if (!ok) break;
        umma_commit_to(smem_addr(acc_full));
        umma_commit_to(acc_full_peer);
      }
    }
  } else if (warp < kFirstEpilogueWarp) {
    // prologue: lane quarter q = warp % 4 (tensor memory is reachable by the
    // warps of that quarter only); thread = row 32 q + lane, the slice's two
    // K halves in turn
    const int q = warp & 3;
    const int prow = q * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(q * 32) << 16;
    auto score_of = [&](int tile) {
      if (tile >= total) return 0.0f;
      const Tile t = decode_tile(tb, a.E, a.n_tiles, tile, rank);
      const int row = t.row0 + prow;
      return row < t.real_end ? __ldg(a.recv_w + row) : 0.0f;
    };
    float next_score = score_of(pair);
    int it = 0;
    for (int tile = pair; tile < total && ok; tile += npairs) {
      const float score = next_score;
      next_score = score_of(tile + npairs);
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int sa = it % kStagesA, s = it % kStages;
        // each lane waits itself (acquiring the copy); the warp leaves together
        bool got = wait_phase(&full_a[sa], (it / kStagesA) & 1u, a.wait_ns);
        if (got && it >= kStages)
          got = wait_phase(&empty[s], ((it / kStages) & 1u) ^ 1u, a.wait_ns);
        got = __all_sync(0xffffffffu, got);
        if (got) {
          tc_fence_after();
          // 16-byte chunk c of row r sits at r * 128 + ((c ^ (r % 8)) * 16); K
          // half kh is chunks 4 kh .. 4 kh + 3 (eight rows of a phase hit eight
          // distinct banks)
          const uint8_t* line = sA + sa * kABytes + prow * 128;
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            uint32_t packed[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int chunk = kh * 4 + c;
              const uint4 v =
                  *reinterpret_cast<const uint4*>(line + ((chunk ^ (prow & 7)) << 4));
              const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float lo = __fmul_rn(__uint_as_float(u[j] << 16), score);
                const float hi = __fmul_rn(__uint_as_float(u[j] & 0xffff0000u), score);
                packed[c * 4 + j] = pack_bf16x2(lo, hi);
              }
            }
            tmem_st16(tmem_a + lane_bits + s * kACols + kh * 16, packed);
          }
          tc_fence_before();
        }
        // the CTA's prologue warps meet once per slice (every one of them,
        // also after a wait that gave up: then all leave together); one
        // thread then frees the h slot (the loads it held are consumed) and
        // tells the even CTA's MMA that this CTA's A stage is in place
        if (!bar_and(got, 1, 32 * kPrologueWarps)) {
          ok = false;
          break;
        }
        if (warp == kFirstPrologueWarp && lane == 0) {
          mbar_arrive(&free_a[sa]);
          mbar_arrive_cluster(cluster_addr(&full[s], 0));
        }
      }
    }
  } else {
    // epilogue: lane quarter q = warp % 4 (tile rows 32 q + lane), column half
    // ch of the accumulator
    const int q = warp & 3;
    const int ch = (warp - kFirstEpilogueWarp) >> 2;
    int n = 0;
    for (int tile = pair; tile < total && ok; tile += npairs, ++n) {
      const Tile ti = decode_tile(tb, a.E, a.n_tiles, tile, rank);
      if (!__all_sync(0xffffffffu, wait_phase(acc_full, n & 1u, a.wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int row = ti.row0 + q * 32 + lane;
      const bool real = row < ti.real_end;
      const bool pad = !real && row < ti.seg_end;
#pragma unroll 1
      for (int j = 0; j < kHalves; ++j) {
        // this warp's kMmaN / 2 columns of column half j, first output column c0
        const int c0 = ti.nt * kBN + j * kMmaN + ch * (kMmaN / 2);
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + j * kMmaN + ch * (kMmaN / 2);
        // the row's columns as bf16 pairs in registers, so the half is handed
        // back to the MMAs before the (slower) stores to HBM
        uint32_t packed[kMmaN / 4];
#pragma unroll
        for (int c = 0; c < kMmaN / 2 / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(taddr + c * 16, v);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            packed[c * 8 + u] =
                real ? pack_bf16x2(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1])) : 0u;
        }
        tc_fence_before();  // the loads above precede the MMAs that reuse the columns
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(&acc_empty[j], 0));
        if (real || pad) {
          __nv_bfloat16* dst = a.y + static_cast<size_t>(row) * a.H + c0;
#pragma unroll
          for (int u = 0; u < kMmaN / 2 / 8; ++u) {
            if (c0 + u * 8 >= a.H) break;  // the last tile's columns past H
            Vec16 o;
            o.u[0] = packed[4 * u];
            o.u[1] = packed[4 * u + 1];
            o.u[2] = packed[4 * u + 2];
            o.u[3] = packed[4 * u + 3];
            st_vec(dst + u * 8, o);
          }
        }
      }
    }
  }
  if (!ok) raise_flag(a.flags, MOE_DEVERR_TIMEOUT);
  tc_fence_before();
  // neither CTA leaves while the other may still reach its shared memory or
  // tensor memory
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    // every MMA must be complete before the columns are released: wait for
    // the last tile's accumulator commit (on the normal path the epilogue
    // already has, and this returns at once)
    if (lane == 0 && my_tiles > 0 &&
        !wait_phase(acc_full, (my_tiles - 1) & 1u, a.wait_ns))
      raise_flag(a.flags, MOE_DEVERR_TIMEOUT);
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// 2-D bf16 tensor map of a row-major [rows, cols] matrix, box [box_rows, kBK]
// with the 128-byte swizzle; out-of-range elements read as zero.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t prepare_w2_kernel() {
  return cudaFuncSetAttribute(w2_absorbed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes));
}

bool w2_shape_ok(int I, int H) {
  return I >= 8 && I % 8 == 0 && H >= kHMultiple && H % kHMultiple == 0;
}

cudaError_t launch_w2_absorbed(const moe_handle* h, const void* hrows, int I, const float* recv_w,
                               const void* w2, int H, void* y, cudaStream_t s) {
  const moe_config& c = h->cfg;
  const int E = c.num_experts;
  const long long rows_cap = static_cast<long long>(h->T) * c.top_k +
                             static_cast<long long>(E) * (h->pad - 1);
  if (rows_cap <= 0) return cudaSuccess;
  if (static_cast<long long>(E) * H > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap tm_h, tm_w2;
  if (!encode_rows(&tm_h, hrows, static_cast<uint64_t>(rows_cap), I, kBM) ||
      !encode_rows(&tm_w2, w2, static_cast<uint64_t>(E) * H, I, kSubRows))
    return cudaErrorInvalidValue;
  W2Args a;
  a.recv_w = recv_w;
  a.off_e = h->off_e;
  a.cnt_e = h->cnt_e;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.flags = h->flags;
  a.wait_ns = h->wait_ns;
  a.rows = static_cast<int>(rows_cap);
  a.E = E;
  a.I = I;
  a.H = H;
  a.n_tiles = (H + kBN - 1) / kBN;
  // sum over experts of ceil(ceil(segment / kBM) / 2) <= pair tiles below
  const long long m_tiles = (rows_cap + static_cast<long long>(E) * (kBM - 1)) / kBM;
  const long long pair_tiles = ((m_tiles + E) / 2) * a.n_tiles;
  if (pair_tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  // CTA pairs in clusters of two, as many as can be resident at once (one
  // CTA per SM: the rings fill its shared memory), never more than there
  // can be pair tiles
  static int max_pairs[64] = {0};
  const int dev = h->device >= 0 && h->device < 64 ? h->device : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs[dev] == 0) {
    cfg.gridDim = dim3(2 * (h->num_sms / 2), 1, 1);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, w2_absorbed_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_pairs[dev] = n;
  }
  const long long pairs = pair_tiles < max_pairs[dev] ? pair_tiles : max_pairs[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (pairs < 1 ? 1 : pairs)), 1, 1);
  return cudaLaunchKernelEx(&cfg, w2_absorbed_kernel, tm_h, tm_w2, a);
}

}  // namespace moe
