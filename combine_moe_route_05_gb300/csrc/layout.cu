// Dispatch layout on the device (sm_103a), with no host synchronisation:
// per-expert and per-virtual-rank counts and offsets, the expert-grouped
// receive layout (stable by token, then k) and the token-deduplicated
// rank-major send layout (one row per (token, rank), stable by token).
// DeepSpeed "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", "Why": a token is sent once per destination rank, arrivals are
// grouped by expert; "Avoid collective token preparation for AutoEP DeepEP",
// "Summary": no argsort and no device-to-host split materialisation.
//
// Tiles of MOE_LAYOUT_TILE_TOKENS tokens, one block per tile and one thread
// per token.  When every tile's block can be resident at once, the whole
// layout is one cooperative launch (layout_scatter_kernel<true>): each block
// marks, in shared-memory bitmasks, which of its tokens use each expert and
// each rank (atomicOr is order-free, so the result does not depend on thread
// timing), publishes its tile's column counts and arrives on an atomic
// ticket; the last block to arrive bumps an epoch the others wait for; then
// every block reads all tiles' counts (its tile bases and the column totals)
// and places its tile with the masks still in shared memory.  Otherwise two
// launches:
//   1. count: each block marks its tile, writes the column counts, and the
//      block that arrives last (an atomic ticket, no waiting) scans them into
//      per-tile bases, counts and offsets;
//   2. scatter: each block rebuilds its bitmasks.
// Placement, in both: the rank of a token among the tile's users of a column
// (expert or rank) is a popcount of the mask bits before it, so every
// position is a pure function of idx (bit-identical on replay).  The tile's
// entries are counting-sorted in shared memory by column (slot = the
// column's segment start in the tile + the entry's rank), and the
// receive-row and send-row outputs are then copied out as one contiguous run
// of rows per column.
//
// Masks are stored word-major with an odd row stride ([word][col], stride
// cols | 1) so that the lanes of a warp, which share a word index and differ in
// column, hit different shared-memory banks.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTile = MOE_LAYOUT_TILE_TOKENS;
constexpr int kWords = kTile / 32;  // mask words per column
constexpr int kThreads = kTile;
static_assert(kTile % 32 == 0 && kTile <= 1024, "tile must be whole warps of one block");

struct LayoutArgs {
  const int32_t* idx;
  int T, K, E, R, epr, ntiles;
  int pad;       // receive segments rounded up to a multiple of pad rows
  int recv_cap;  // receive rows: T*K + E*(pad-1)
  uint32_t* flags;
  // arrivals of the tile hand-over (low 32 bits) and its epoch (high 32 bits)
  unsigned long long* ticket;
  unsigned long long wait_ns;  // limit of the single-pass kernel's wait for the epoch
  int32_t* cnt_e;
  int32_t* off_e;
  int32_t* cnt_send_r;
  int32_t* off_send_r;
  int32_t* cnt_recv_r;
  int32_t* off_recv_r;
  int32_t* S;
  int32_t* pos;
  int32_t* recv_token;
  int32_t* recv_k;
  int32_t* send_token;
  int32_t* send_row_of;
  int32_t* recv_send_row;
  int32_t* tile_hist;  // [ntiles][cols] tile counts (exclusive tile bases after
                       // the two-launch path's scan)
};

__host__ __device__ constexpr int col_stride(int cols) { return cols | 1; }

// Fills rank_of[e] = e / epr (shared memory, all threads of the block).
__device__ __forceinline__ void fill_rank_table(const LayoutArgs& a, int32_t* rank_of) {
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) rank_of[e] = e / a.epr;
}

// Loads the experts of this thread's token t (if t < T) into ek; issued
// before the shared-memory set-up so that its latency overlaps it.
__device__ __forceinline__ void load_token(const LayoutArgs& a, int t, int (&ek)[MOE_MAX_TOPK]) {
  if (t >= a.T) return;
  const int32_t* row = a.idx + static_cast<size_t>(t) * a.K;
#pragma unroll
  for (int k = 0; k < MOE_MAX_TOPK; ++k) {
    if (k >= a.K) break;
    ek[k] = __ldg(row + k);
  }
}

// Validates this thread's token t (experts in ek, from load_token) and sets
// its bits in the tile's expert and rank masks (rank_of: the expert -> rank
// table).  Returns the valid-entry bitmask.
__device__ __forceinline__ uint32_t mark_token(const LayoutArgs& a, int t, uint32_t* masks, int cp,
                                               const int32_t* rank_of,
                                               const int (&ek)[MOE_MAX_TOPK]) {
  uint32_t valid = 0;
  if (t >= a.T) return 0;
  const int word = threadIdx.x >> 5;
  const uint32_t bit = 1u << (threadIdx.x & 31);
  uint32_t bad = 0;
#pragma unroll
  for (int k = 0; k < MOE_MAX_TOPK; ++k) {
    if (k >= a.K) break;
    const int e = ek[k];
    bool ok = e >= 0 && e < a.E;
    if (!ok) bad |= MOE_DEVERR_BAD_EXPERT;
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      if (j >= k) break;
      if (ok && ((valid >> j) & 1u) && ek[j] == e) {
        ok = false;
        bad |= MOE_DEVERR_DUP_EXPERT;
      }
    }
    if (ok) {
      valid |= 1u << k;
      atomicOr(&masks[word * cp + e], bit);
      atomicOr(&masks[word * cp + a.E + rank_of[e]], bit);
    }
  }
  if (bad) raise_flag(a.flags, bad);
  return valid;
}

// Exclusive scan, in place, of v[0, n) (n <= 4 * kThreads) by the whole
// block: each thread a run of up to four entries, a warp scan of the runs'
// sums, and a scan of the warps' totals.  `ws`: kThreads / 32 + 1 ints of
// shared memory.  Ends with a barrier.
__device__ void block_scan(int32_t* v, int n, int32_t* ws) {
  constexpr int kWarps = kThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (n + kThreads - 1) / kThreads;  // 1 .. 4
  const int i0 = per * threadIdx.x;
  int x[4];
  int s = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[j] = j < per && i0 + j < n ? v[i0 + j] : 0;
    s += x[j];
  }
  int incl = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < kWarps ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += o;
    }
    if (lane < kWarps) ws[lane] = wi - w;
  }
  __syncthreads();
  int run = ws[warp] + incl - s;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < per && i0 + j < n) v[i0 + j] = run;
    run += x[j];
  }
  __syncthreads();
}

// Column values c[0, E) and c[E, E + R) scanned into the split form
// o[0..E] | o[E+1..E+R+1]: experts then ranks, each from zero, each with its
// total at the end (o: E + R + 2 ints of shared memory, which may be c's own
// split slots).  Expert values are rounded up to a multiple of `pad` first.
// Ends with a barrier.
__device__ void scan_split(const LayoutArgs& a, int32_t* o, int pad, int32_t* ws) {
  const int cols = a.E + a.R;
  if (pad > 1)
    for (int e = threadIdx.x; e < a.E; e += kThreads) o[e] = (o[e] + pad - 1) / pad * pad;
  if (threadIdx.x == 0) {
    o[a.E] = 0;
    o[cols + 1] = 0;
  }
  __syncthreads();
  block_scan(o, cols + 2, ws);
  // the rank entries continue the expert scan: restart them at zero
  const int tot_e = o[a.E];
  for (int j = a.E + 1 + threadIdx.x; j < cols + 2; j += kThreads) o[j] -= tot_e;
  __syncthreads();
}

// Exclusive scans of the column totals, tot[0, E) (expert segments rounded up
// to the padding) and tot[E, E + R) (ranks), into off[0..E] (off_e) and
// off[E+1..E+R+1] (off_s), shared memory.  With `publish`, also writes the
// layout's count and offset arrays and S.  Ends with a barrier.
__device__ void scan_totals(const LayoutArgs& a, const int32_t* tot, int32_t* off, int32_t* ws,
                            bool publish) {
  const int cols = a.E + a.R;
  for (int c = threadIdx.x; c < cols; c += kThreads) off[c + (c >= a.E ? 1 : 0)] = tot[c];
  scan_split(a, off, a.pad, ws);
  if (publish) {
    const int32_t* off_s = off + a.E + 1;
    for (int e = threadIdx.x; e < a.E; e += kThreads) {
      a.cnt_e[e] = tot[e];
      a.off_e[e] = off[e];
    }
    for (int r = threadIdx.x; r < a.R; r += kThreads) {
      a.cnt_send_r[r] = tot[a.E + r];
      a.off_send_r[r] = off_s[r];
      // rows that arrive at rank r (pads excluded); its region starts at the
      // padded offset of its first expert
      int n = 0;
      for (int e = r * a.epr; e < (r + 1) * a.epr; ++e) n += tot[e];
      a.off_recv_r[r] = off[r * a.epr];
      a.cnt_recv_r[r] = n;
    }
    if (threadIdx.x == 0) {
      a.off_e[a.E] = off[a.E];
      a.off_send_r[a.R] = off_s[a.R];
      *a.S = off_s[a.R];
      a.off_recv_r[a.R] = off[a.E];
    }
  }
}

// The last block of the two-launch path: exclusive scan of each column over
// the tiles (in place in tile_hist), then the scans of the column totals.
// `scratch`: 2 (E + R) + 2 + kThreads / 32 + 1 ints of shared memory.
__device__ void scan_tiles(const LayoutArgs& a, int32_t* scratch) {
  const int cols = a.E + a.R;
  int32_t* tot = scratch;
  for (int col = threadIdx.x; col < cols; col += kThreads) {
    int run = 0;
    for (int t0 = 0; t0 < a.ntiles; t0 += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        v[i] = t0 + i < a.ntiles ? __ldcg(a.tile_hist + static_cast<size_t>(t0 + i) * cols + col) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (t0 + i < a.ntiles) a.tile_hist[static_cast<size_t>(t0 + i) * cols + col] = run;
        run += v[i];
      }
    }
    tot[col] = run;
  }
  __syncthreads();
  scan_totals(a, tot, scratch + cols, scratch + 2 * cols + 2, true);
}

__global__ void __launch_bounds__(kThreads, 1) layout_count_kernel(LayoutArgs a) {
  extern __shared__ uint32_t lsm[];
  const int cols = a.E + a.R;
  const int cp = col_stride(cols);
  uint32_t* masks = lsm;  // [kWords][cp]
  int32_t* rank_of = reinterpret_cast<int32_t*>(lsm + kWords * cp);  // [E]
  const int tile = blockIdx.x;
  int ek[MOE_MAX_TOPK];
  load_token(a, tile * kTile + threadIdx.x, ek);
  for (int i = threadIdx.x; i < kWords * cp; i += kThreads) masks[i] = 0;
  fill_rank_table(a, rank_of);
  __syncthreads();
  mark_token(a, tile * kTile + threadIdx.x, masks, cp, rank_of, ek);
  __syncthreads();
  for (int col = threadIdx.x; col < cols; col += kThreads) {
    int c = 0;
#pragma unroll 8
    for (int w = 0; w < kWords; ++w) c += __popc(masks[w * cp + col]);
    a.tile_hist[static_cast<size_t>(tile) * cols + col] = c;
  }
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) {
    __threadfence();  // the tile's counts before its arrival
    is_last = static_cast<uint32_t>(atomicAdd(a.ticket, 1ull)) == static_cast<uint32_t>(a.ntiles - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  scan_tiles(a, reinterpret_cast<int32_t*>(masks));  // masks are dead now (16 (E + R + 1) ints)
  // ready for the next layout: arrivals back to zero, the epoch advanced
  if (threadIdx.x == 0) atomicAdd(a.ticket, (1ull << 32) - static_cast<unsigned long long>(a.ntiles));
}

// shared memory of the scatter kernel, in order
struct ScatterSmem {
  int cols, cp, K, KR, E;  // KR = min(K, R): send entries per token at most
  // the masks, and after the token pass the tile's positions [kTile][K]
  __host__ __device__ size_t masks() const { return 0; }
  __host__ __device__ size_t masks_bytes() const {
    const size_t m = sizeof(uint32_t) * kWords * cp, p = sizeof(int32_t) * kTile * K;
    return m > p ? m : p;
  }
  __host__ __device__ size_t pre() const { return masks() + masks_bytes(); }
  __host__ __device__ size_t seg() const { return align(pre() + sizeof(uint16_t) * kWords * cp); }
  __host__ __device__ size_t srow() const { return seg() + sizeof(int32_t) * (cols + 2); }
  __host__ __device__ size_t rst() const { return srow() + sizeof(int32_t) * kTile * K; }
  __host__ __device__ size_t sst() const { return rst() + sizeof(uint32_t) * kTile * K; }
  __host__ __device__ size_t base() const { return sst() + sizeof(uint32_t) * kTile * KR; }
  __host__ __device__ size_t off() const { return base() + sizeof(int32_t) * cols; }
  __host__ __device__ size_t rank_of() const { return off() + sizeof(int32_t) * (cols + 2); }
  __host__ __device__ size_t tot() const { return rank_of() + sizeof(int32_t) * E; }
  __host__ __device__ size_t ws() const { return tot() + sizeof(int32_t) * cols; }
  // the column totals (single pass) and the block scan's warp sums
  __host__ __device__ size_t bytes() const { return ws() + sizeof(int32_t) * (kThreads / 32 + 1); }
  __host__ __device__ static size_t align(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }
};

// packed staging entries (expert < 512, k < 16, token in tile < 1024)
__device__ __forceinline__ uint32_t pack_recv(int e, int k, int tl) {
  return static_cast<uint32_t>(e) | (static_cast<uint32_t>(k) << 9) | (static_cast<uint32_t>(tl) << 13);
}
__device__ __forceinline__ uint32_t pack_send(int r, int tl) {
  return static_cast<uint32_t>(r) | (static_cast<uint32_t>(tl) << 9);
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// kSinglePass = false: the second of two launches (the counts and their
// scan come from layout_count_kernel).  kSinglePass = true: the whole layout
// in one cooperative launch (all tiles resident at once): each block counts
// its tile and arrives; the last block to arrive bumps an epoch that the
// other blocks wait for (at most wait_ns, 1 s unless the handle sets another
// limit, then the status word's time-out bit and no writes); every block then derives its tile bases and the column offsets
// from all tiles' counts and places its tile with the masks still in shared
// memory.
template <bool kSinglePass>
__global__ void __launch_bounds__(kThreads, 1) layout_scatter_kernel(LayoutArgs a) {
  if (kSinglePass) grid_dependency_wait();
  extern __shared__ __align__(16) uint8_t ssm[];
  const int cols = a.E + a.R;
  const int cp = col_stride(cols);
  const int KR = a.K < a.R ? a.K : a.R;
  const ScatterSmem L{cols, cp, a.K, KR, a.E};
  uint32_t* masks = reinterpret_cast<uint32_t*>(ssm + L.masks());  // [kWords][cp]
  uint16_t* pre = reinterpret_cast<uint16_t*>(ssm + L.pre());      // [kWords][cp]
  int32_t* seg = reinterpret_cast<int32_t*>(ssm + L.seg());        // seg_e[E+1] | seg_r[R+1]
  int32_t* srow_s = reinterpret_cast<int32_t*>(ssm + L.srow());    // [kTile][K]
  uint32_t* rst = reinterpret_cast<uint32_t*>(ssm + L.rst());      // receive entries, by column
  uint32_t* sst = reinterpret_cast<uint32_t*>(ssm + L.sst());      // send entries, by column
  int32_t* base = reinterpret_cast<int32_t*>(ssm + L.base());      // [cols] tile bases
  int32_t* off = reinterpret_cast<int32_t*>(ssm + L.off());        // off_e[E+1] | off_s[R+1]
  int32_t* rank_of = reinterpret_cast<int32_t*>(ssm + L.rank_of()); // [E] expert -> rank
  const int tile = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int tile_t0 = tile * kTile;
  const int tile_n = max(0, min(kTile, a.T - tile_t0));  // tokens in this tile

  const int t = tile_t0 + threadIdx.x;
  int ek[MOE_MAX_TOPK];
  load_token(a, t, ek);
  for (int i = threadIdx.x; i < kWords * cp; i += kThreads) masks[i] = 0;
  fill_rank_table(a, rank_of);
  auto load_bases = [&]() {
    for (int c = threadIdx.x; c < cols; c += kThreads) {
      base[c] = __ldcg(a.tile_hist + static_cast<size_t>(tile) * cols + c);
      off[c + (c >= a.E ? 1 : 0)] = c < a.E ? __ldcg(a.off_e + c) : __ldcg(a.off_send_r + c - a.E);
    }
    if (threadIdx.x == 0) {
      off[a.E] = __ldcg(a.off_e + a.E);
      off[cols + 1] = __ldcg(a.off_send_r + a.R);
    }
  };
  if (!kSinglePass) load_bases();
  __syncthreads();
  const uint32_t valid = mark_token(a, t, masks, cp, rank_of, ek);
  __syncthreads();
  // the tile's column counts (the single pass publishes them at once)
  for (int col = threadIdx.x; col < cols; col += kThreads) {
    int run = 0;
#pragma unroll 8
    for (int w = 0; w < kWords; ++w) run += __popc(masks[w * cp + col]);
    seg[col + (col >= a.E ? 1 : 0)] = run;
    if (kSinglePass) a.tile_hist[static_cast<size_t>(tile) * cols + col] = run;
  }
  __syncthreads();
  // grid-wide hand-over of the tile counts (single pass): one 64-bit word
  // holds the arrivals and the epoch; the last block to arrive resets the
  // arrivals and advances the epoch in one atomic, the others wait for the
  // epoch below, after the work that does not need the other tiles
  __shared__ uint32_t epoch0;
  __shared__ int last, failed;
  if (kSinglePass && threadIdx.x == 0) {
    __threadfence();  // the tile's counts before its arrival
    const unsigned long long old = atomicAdd(a.ticket, 1ull);
    epoch0 = static_cast<uint32_t>(old >> 32);
    last = static_cast<uint32_t>(old) == static_cast<uint32_t>(a.ntiles - 1);
    failed = 0;
    if (last) {
      __threadfence();
      atomicAdd(a.ticket, (1ull << 32) - static_cast<unsigned long long>(a.ntiles));
    }
  }
  // exclusive prefix of the popcounts over the words of each column, and the
  // tile's column offsets (experts, ranks)
  for (int col = threadIdx.x; col < cols; col += kThreads) {
    int run = 0;
#pragma unroll 8
    for (int w = 0; w < kWords; ++w) {
      pre[w * cp + col] = static_cast<uint16_t>(run);
      run += __popc(masks[w * cp + col]);
    }
  }
  int32_t* ws = reinterpret_cast<int32_t*>(ssm + L.ws());
  scan_split(a, seg, 1, ws);

  if (kSinglePass) {
    if (threadIdx.x == 0 && !last) {
      const unsigned long long t0 = global_ns();
      while (static_cast<uint32_t>(ld_acquire_u64(a.ticket) >> 32) == epoch0) {
        if (global_ns() - t0 > a.wait_ns) {
          raise_flag(a.flags, MOE_DEVERR_TIMEOUT);
          failed = 1;
          break;
        }
      }
    }
    __syncthreads();
    if (failed) return;
    // per column: the counts of the tiles before this one (its base) and of
    // all tiles (the column total), 16 loads in flight per thread; where a
    // column has several threads (kThreads / cols of them), they take
    // alternate tiles and add up in shared memory
    int32_t* tot = reinterpret_cast<int32_t*>(ssm + L.tot());
    const int per = cols <= kThreads ? kThreads / cols : 1;
    for (int c = threadIdx.x; c < cols; c += kThreads) {
      base[c] = 0;
      tot[c] = 0;
    }
    __syncthreads();
    if (threadIdx.x < per * cols || per == 1) {
      const int part = per == 1 ? 0 : threadIdx.x / cols;
      for (int col = per == 1 ? threadIdx.x : threadIdx.x % cols; col < cols; col += kThreads) {
        int before = 0, all = 0;
        for (int t0 = part; t0 < a.ntiles; t0 += 16 * per) {
          int v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tt = t0 + i * per;
            v[i] = tt < a.ntiles ? __ldcg(a.tile_hist + static_cast<size_t>(tt) * cols + col) : 0;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (t0 + i * per < tile) before += v[i];
            all += v[i];
          }
        }
        if (per == 1) {
          base[col] = before;
          tot[col] = all;
        } else {
          atomicAdd(&base[col], before);
          atomicAdd(&tot[col], all);
        }
      }
    }
    __syncthreads();
    // offsets in shared memory; block 0 also publishes the count arrays
    scan_totals(a, tot, off, ws, tile == 0);
  }

  // base[c] becomes the first global row of this tile's run of column c
  for (int c = threadIdx.x; c < cols; c += kThreads) base[c] += c < a.E ? off[c] : off[c + 1];
  __syncthreads();
  const int32_t* off_e = off;
  const int32_t* tot_s = reinterpret_cast<const int32_t*>(ssm + L.tot());  // single pass only
  const int32_t* seg_e = seg;
  const int32_t* seg_r = seg + a.E + 1;
  const int n_recv_rows = a.recv_cap;
  const int n_send_rows = a.T * KR;
  const uint32_t lt = lanemask_lt();

  // token pass: positions, and the tile's counting sort into the staging
  // arrays (an entry's slot is its column's segment start plus its rank)
  int pk[MOE_MAX_TOPK];  // this token's positions, staged for a coalesced copy-out
  if (t < a.T) {
    int rk[MOE_MAX_TOPK];  // rank of each valid entry's expert
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k) {
      if (k >= a.K) break;
      int p = -1, srow = -1;
      if ((valid >> k) & 1u) {
        const int e = ek[k];
        const int r = rank_of[e];
        rk[k] = r;
        const int ce = warp * cp + e;
        const int cr = warp * cp + a.E + r;
        const int rank_e = pre[ce] + __popc(masks[ce] & lt);
        const int rank_r = pre[cr] + __popc(masks[cr] & lt);
        p = base[e] + rank_e;
        srow = base[a.E + r] + rank_r;
        // the scan guarantees p < T*K and srow < S; a violation (inconsistent
        // counts) is reported and the entry dropped instead of written
        if (p < 0 || p >= n_recv_rows || srow < 0 || srow >= n_send_rows) {
          raise_flag(a.flags, MOE_DEVERR_INTERNAL);
          p = -1;
          srow = -1;
        } else {
          rst[seg_e[e] + rank_e] = pack_recv(e, k, threadIdx.x);
          bool first = true;
#pragma unroll
          for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            if (j >= k) break;
            if (((valid >> j) & 1u) && rk[j] == r) first = false;
          }
          if (first) sst[seg_r[r] + rank_r] = pack_send(r, threadIdx.x);
        }
      }
      pk[k] = p;
      srow_s[threadIdx.x * a.K + k] = srow;
    }
  }
  __syncthreads();
  // the masks are dead: their space takes the positions
  int32_t* pos_s = reinterpret_cast<int32_t*>(ssm + L.masks());
  if (t < a.T) {
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k) {
      if (k >= a.K) break;
      pos_s[threadIdx.x * a.K + k] = pk[k];
    }
  }
  __syncthreads();

  // copy-out, one loop so that each thread has the stores of all three kinds
  // in flight: pos and send_row_of (token-major, contiguous for the tile),
  // receive entries and send entries (each a run of consecutive rows per
  // column)
  {
    const int n = tile_n * a.K;
    const int n_recv = seg_e[a.E], n_send = seg_r[a.R];
    const int n_all = max(n, max(n_recv, n_send));
    int32_t* pos_g = a.pos + static_cast<size_t>(tile_t0) * a.K;
    int32_t* srow_g = a.send_row_of + static_cast<size_t>(tile_t0) * a.K;
    for (int i = threadIdx.x; i < n_all; i += kThreads) {
      if (i < n) {
        pos_g[i] = pos_s[i];
        srow_g[i] = srow_s[i];
      }
      if (i < n_recv) {
        const uint32_t u = rst[i];
        const int e = u & 511u, k = (u >> 9) & 15u, tl = u >> 13;
        // a slot left empty by a dropped inconsistent entry holds stale data
        const int row = e < a.E ? base[e] + (i - seg_e[e]) : -1;
        if (e >= a.E || k >= a.K || tl >= tile_n || row < 0 || row >= n_recv_rows) {
          raise_flag(a.flags, MOE_DEVERR_INTERNAL);
        } else {
          a.recv_token[row] = tile_t0 + tl;
          a.recv_k[row] = k;
          a.recv_send_row[row] = srow_s[tl * a.K + k];
        }
      }
      if (i < n_send) {
        const uint32_t u = sst[i];
        const int r = u & 511u, tl = u >> 9;
        const int row = r < a.R ? base[a.E + r] + (i - seg_r[r]) : -1;
        if (tl >= tile_n || row < 0 || row >= n_send_rows) {
          raise_flag(a.flags, MOE_DEVERR_INTERNAL);
        } else {
          a.send_token[row] = tile_t0 + tl;
        }
      }
    }
  }

  // pad rows of the expert segments (this block takes experts blockIdx.x,
  // blockIdx.x + gridDim.x, ...), then the tails: receive rows past off_e[E]
  // and send rows past S
  if (a.pad > 1) {
    for (int e = blockIdx.x; e < a.E; e += gridDim.x) {
      const int lo = off_e[e] + (kSinglePass ? tot_s[e] : __ldcg(a.cnt_e + e)), hi = off_e[e + 1];
      for (int p = lo + threadIdx.x; p < hi; p += kThreads) {
        a.recv_token[p] = -1;
        a.recv_k[p] = -1;
        a.recv_send_row[p] = -1;
      }
    }
  }
  const long long gtid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const long long gsize = static_cast<long long>(gridDim.x) * kThreads;
  for (long long p = off[a.E] + gtid; p < n_recv_rows; p += gsize) {
    a.recv_token[p] = -1;
    a.recv_k[p] = -1;
    a.recv_send_row[p] = -1;
  }
  for (long long s = off[cols + 1] + gtid; s < n_send_rows; s += gsize) a.send_token[s] = -1;
}

size_t count_smem(int cols, int E) {
  return (static_cast<size_t>(kWords) * col_stride(cols) + E) * sizeof(uint32_t);
}

size_t scatter_smem(int cols, int K, int R) {
  return ScatterSmem{cols, col_stride(cols), K, K < R ? K : R, cols - R}.bytes();
}

}  // namespace

size_t layout_smem_bytes(int E, int R) {
  const size_t a = count_smem(E + R, E), b = scatter_smem(E + R, MOE_MAX_TOPK, R);
  return a > b ? a : b;
}

cudaError_t prepare_layout_kernels() {
  const int max_smem = static_cast<int>(layout_smem_bytes(MOE_MAX_EXPERTS, MOE_MAX_EXPERTS));
  cudaError_t e = cudaFuncSetAttribute(layout_count_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(layout_scatter_kernel<false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(layout_scatter_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

int layout_tiles(int T) { return T > 0 ? (T + kTile - 1) / kTile : 1; }

namespace {
// Blocks of the single-pass kernel that fit on the current device at once
// for a given shared-memory size (0 if the query fails); cached, since the
// layout is launched every step.
int resident_single_pass_blocks(size_t smem) {
  struct Entry {
    int dev;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].smem == smem) return cache[i].blocks;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layout_scatter_kernel<true>, kThreads,
                                                    smem) != cudaSuccess)
    return 0;
  const int blocks = per_sm * sms;
  if (used < 16) cache[used++] = Entry{dev, smem, blocks};
  return blocks;
}
}  // namespace

// The two launches over caller-chosen buffers: the outputs in `out`, the
// status word `flags` (may be null), and the scratch (arrival ticket, zero on
// entry, and tiles * (E + R) tile counters).
cudaError_t launch_layout_buffers(const moe_config& c, const int32_t* idx, int T,
                                  const moe_layout& out, uint32_t* flags, uint32_t* ticket,
                                  int32_t* tile_hist, int max_tiles, unsigned long long wait_ns,
                                  cudaStream_t s) {
  LayoutArgs a;
  a.idx = idx;
  a.T = T;
  a.K = c.top_k;
  a.E = c.num_experts;
  a.R = c.num_ranks;
  a.epr = c.num_experts / c.num_ranks;
  a.ntiles = layout_tiles(T);
  if (a.ntiles > max_tiles) return cudaErrorInvalidValue;
  a.pad = c.pad_align > 1 ? c.pad_align : 1;
  a.recv_cap = T * a.K + a.E * (a.pad - 1);
  a.flags = flags;
  a.ticket = reinterpret_cast<unsigned long long*>(ticket);
  a.wait_ns = wait_ns;
  a.cnt_e = out.cnt_e;
  a.off_e = out.off_e;
  a.cnt_send_r = out.cnt_send_r;
  a.off_send_r = out.off_send_r;
  a.cnt_recv_r = out.cnt_recv_r;
  a.off_recv_r = out.off_recv_r;
  a.S = out.S;
  a.pos = out.pos;
  a.recv_token = out.recv_token;
  a.recv_k = out.recv_k;
  a.send_token = out.send_token;
  a.send_row_of = out.send_row_of;
  a.recv_send_row = out.recv_send_row;
  a.tile_hist = tile_hist;
  const int cols = a.E + a.R;
  // one cooperative launch when every tile's block can be resident at once
  // (the blocks wait for the last one's scan), else two launches
  const size_t one_smem = scatter_smem(cols, a.K, a.R);
  if (a.ntiles <= resident_single_pass_blocks(one_smem)) {
    const cudaError_t e =
        launch_chained(layout_scatter_kernel<true>, dim3(a.ntiles), dim3(kThreads), one_smem, s, true, a);
    if (e == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();  // not launched: take the two-launch path
  }
  layout_count_kernel<<<a.ntiles, kThreads, count_smem(cols, a.E), s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  layout_scatter_kernel<false><<<a.ntiles, kThreads, scatter_smem(cols, a.K, a.R), s>>>(a);
  return cudaGetLastError();
}

int layout_launches(const moe_config& c, int T) {
  const int cols = c.num_experts + c.num_ranks;
  const size_t one_smem = scatter_smem(cols, c.top_k, c.num_ranks);
  return layout_tiles(T) <= resident_single_pass_blocks(one_smem) ? 1 : 2;
}

cudaError_t launch_layout(const moe_handle* h, const int32_t* idx, int T, cudaStream_t s) {
  moe_layout out{};
  out.cnt_e = h->cnt_e;
  out.off_e = h->off_e;
  out.cnt_send_r = h->cnt_send_r;
  out.off_send_r = h->off_send_r;
  out.cnt_recv_r = h->cnt_recv_r;
  out.off_recv_r = h->off_recv_r;
  out.S = h->S;
  out.pos = h->pos;
  out.recv_token = h->recv_token;
  out.recv_k = h->recv_k;
  out.send_token = h->send_token;
  out.send_row_of = h->send_row_of;
  out.recv_send_row = h->recv_send_row;
  return launch_layout_buffers(h->cfg, idx, T, out, h->flags, h->ticket, h->tile_hist,
                               h->max_tiles, h->wait_ns, s);
}

}  // namespace moe
