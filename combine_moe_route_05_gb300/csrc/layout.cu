// Dispatch layout on the device (sm_103a), with no host synchronisation:
// per-expert and per-virtual-rank counts and offsets, the expert-grouped
// receive layout (stable by token, then k) and the token-deduplicated
// rank-major send layout (one row per (token, rank), stable by token).
// DeepSpeed "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", "Why": a token is sent once per destination rank, arrivals are
// grouped by expert; "Avoid collective token preparation for AutoEP DeepEP",
// "Summary": no argsort and no device-to-host split materialisation.
//
// Two launches over tiles of 1024 tokens (one token per thread):
//   1. count: each block marks, in shared-memory bitmasks, which of its
//      tokens use each expert and each rank (atomicOr is order-free, so the
//      result does not depend on thread timing), writes per-tile column
//      counts, and the block that arrives last (an atomic ticket, no
//      waiting) scans them into per-tile bases, counts and offsets;
//   2. scatter: each block rebuilds its bitmasks; the rank of a token among
//      the tile's users of an expert is a popcount of the mask words before
//      it, so every position is a pure function of idx (bit-identical on
//      replay).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTile = MOE_LAYOUT_TILE;
constexpr int kWords = kTile / 32;  // mask words per column
constexpr int kThreads = kTile;
constexpr int kWarps = kThreads / 32;

struct LayoutArgs {
  const int32_t* idx;
  int T, K, E, R, epr, ntiles, max_tiles;
  uint32_t* flags;
  uint32_t* ticket;
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
  int32_t* tile_hist;
};

// Loads this thread's token (if any), validates it and sets its bits in the
// tile's expert and rank masks.  Returns the valid-entry bitmask; ek holds the
// expert of each entry.
__device__ __forceinline__ uint32_t mark_token(const LayoutArgs& a, int t, uint32_t* masks,
                                               int (&ek)[MOE_MAX_TOPK]) {
  uint32_t valid = 0;
  if (t >= a.T) return 0;
  const int word = threadIdx.x >> 5;
  const uint32_t bit = 1u << (threadIdx.x & 31);
  const int32_t* row = a.idx + static_cast<size_t>(t) * a.K;
  uint32_t bad = 0;
#pragma unroll
  for (int k = 0; k < MOE_MAX_TOPK; ++k) {
    if (k >= a.K) break;
    const int e = __ldg(row + k);
    ek[k] = e;
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
      atomicOr(&masks[e * kWords + word], bit);
      atomicOr(&masks[(a.E + e / a.epr) * kWords + word], bit);
    }
  }
  if (bad) raise_flag(a.flags, bad);
  return valid;
}

__global__ void __launch_bounds__(kThreads, 1) layout_count_kernel(LayoutArgs a) {
  extern __shared__ uint32_t lsm[];
  uint32_t* masks = lsm;  // [(E+R) * kWords]
  const int cols = a.E + a.R;
  const int tile = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < cols * kWords; i += kThreads) masks[i] = 0;
  __syncthreads();
  int ek[MOE_MAX_TOPK];
  mark_token(a, tile * kTile + threadIdx.x, masks, ek);
  __syncthreads();
  for (int col = warp; col < cols; col += kWarps) {
    const int c = __reduce_add_sync(0xffffffffu, __popc(masks[col * kWords + lane]));
    if (lane == 0) a.tile_hist[static_cast<size_t>(col) * a.max_tiles + tile] = c;
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = atomicAdd(a.ticket, 1u) == static_cast<uint32_t>(a.ntiles - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Last block: exclusive scan of each column over the tiles (in place), then
  // exclusive scans over experts and over ranks.
  int32_t* tot = reinterpret_cast<int32_t*>(masks);  // [cols], masks are dead now
  for (int col = threadIdx.x; col < cols; col += kThreads) {
    int32_t* base = a.tile_hist + static_cast<size_t>(col) * a.max_tiles;
    int run = 0;
    for (int t0 = 0; t0 < a.ntiles; t0 += 16) {
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = t0 + i < a.ntiles ? __ldcg(base + t0 + i) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (t0 + i < a.ntiles) base[t0 + i] = run;
        run += v[i];
      }
    }
    tot[col] = run;
  }
  __syncthreads();
  if (warp < 2) {
    // warp 0 scans the E expert totals, warp 1 the R rank totals
    const int n = warp == 0 ? a.E : a.R;
    const int32_t* src = tot + (warp == 0 ? 0 : a.E);
    int32_t* cnt = warp == 0 ? a.cnt_e : a.cnt_send_r;
    int32_t* off = warp == 0 ? a.off_e : a.off_send_r;
    const int per = (n + 31) / 32;
    const int lo = lane * per, hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += src[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int run = incl - local;
    for (int i = lo; i < hi; ++i) {
      cnt[i] = src[i];
      off[i] = run;
      run += src[i];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      off[n] = total;
      if (warp == 1) *a.S = total;
    }
  }
  __syncthreads();
  __threadfence_block();
  for (int r = threadIdx.x; r < a.R; r += kThreads) {
    const int lo = a.off_e[r * a.epr], hi = a.off_e[(r + 1) * a.epr];
    a.off_recv_r[r] = lo;
    a.cnt_recv_r[r] = hi - lo;
  }
  if (threadIdx.x == 0) {
    a.off_recv_r[a.R] = a.off_e[a.E];
    *a.ticket = 0;  // ready for the next layout
  }
}

__global__ void __launch_bounds__(kThreads, 1) layout_scatter_kernel(LayoutArgs a) {
  extern __shared__ uint32_t lsm[];
  const int cols = a.E + a.R;
  uint32_t* masks = lsm;                                                  // [cols * kWords]
  uint16_t* pre = reinterpret_cast<uint16_t*>(masks + cols * kWords);     // [cols * kWords]
  int32_t* base = reinterpret_cast<int32_t*>(pre + cols * kWords);        // [cols] tile bases
  int32_t* off = base + cols;                                             // [E+1 | R+1]
  const int tile = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < cols * kWords; i += kThreads) masks[i] = 0;
  for (int c = threadIdx.x; c < cols; c += kThreads) {
    base[c] = a.tile_hist[static_cast<size_t>(c) * a.max_tiles + tile];
    off[c + (c >= a.E ? 1 : 0)] = c < a.E ? a.off_e[c] : a.off_send_r[c - a.E];
  }
  if (threadIdx.x == 0) {
    off[a.E] = a.off_e[a.E];
    off[cols + 1] = a.off_send_r[a.R];
  }
  __syncthreads();
  const int t = tile * kTile + threadIdx.x;
  int ek[MOE_MAX_TOPK];
  const uint32_t valid = mark_token(a, t, masks, ek);
  __syncthreads();
  for (int col = warp; col < cols; col += kWarps) {
    const int c = __popc(masks[col * kWords + lane]);
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    pre[col * kWords + lane] = static_cast<uint16_t>(incl - c);
  }
  __syncthreads();

  const int n_recv_rows = a.T * a.K;
  const int n_send_rows = a.T * (a.K < a.R ? a.K : a.R);
  if (t < a.T) {
    const uint32_t lt = lanemask_lt();
    const int32_t* off_e = off;
    const int32_t* off_s = off + a.E + 1;
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k) {
      if (k >= a.K) break;
      const size_t tk = static_cast<size_t>(t) * a.K + k;
      if (!((valid >> k) & 1u)) {
        a.pos[tk] = -1;
        a.send_row_of[tk] = -1;
        continue;
      }
      const int e = ek[k];
      const int ce = e * kWords + warp;
      const int p = off_e[e] + base[e] + pre[ce] + __popc(masks[ce] & lt);
      const int r = e / a.epr;
      const int cr = (a.E + r) * kWords + warp;
      const int srow = off_s[r] + base[a.E + r] + pre[cr] + __popc(masks[cr] & lt);
      // the scan guarantees p < T*K and srow < S; a violation (inconsistent
      // counts) is reported instead of written
      if (p < 0 || p >= n_recv_rows || srow < 0 || srow >= n_send_rows) {
        raise_flag(a.flags, MOE_DEVERR_INTERNAL);
        a.pos[tk] = -1;
        a.send_row_of[tk] = -1;
        continue;
      }
      a.pos[tk] = p;
      a.recv_token[p] = t;
      a.recv_k[p] = k;
      a.send_row_of[tk] = srow;
      a.recv_send_row[p] = srow;
      bool first = true;
#pragma unroll
      for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (j >= k) break;
        if (((valid >> j) & 1u) && ek[j] / a.epr == r) first = false;
      }
      if (first) a.send_token[srow] = t;
    }
  }

  // tails: receive rows past off_e[E] and send rows past S
  const long long gtid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const long long gsize = static_cast<long long>(gridDim.x) * kThreads;
  const long long n_recv = static_cast<long long>(a.T) * a.K;
  for (long long p = off[a.E] + gtid; p < n_recv; p += gsize) {
    a.recv_token[p] = -1;
    a.recv_k[p] = -1;
    a.recv_send_row[p] = -1;
  }
  const long long n_send = static_cast<long long>(a.T) * (a.K < a.R ? a.K : a.R);
  for (long long s = off[cols + 1] + gtid; s < n_send; s += gsize) a.send_token[s] = -1;
}

size_t count_smem(int cols) { return static_cast<size_t>(cols) * kWords * sizeof(uint32_t); }

size_t scatter_smem(int cols) {
  return static_cast<size_t>(cols) * kWords * (sizeof(uint32_t) + sizeof(uint16_t)) +
         static_cast<size_t>(cols) * sizeof(int32_t) + static_cast<size_t>(cols + 2) * sizeof(int32_t);
}

}  // namespace

size_t layout_smem_bytes(int E, int R) {
  const size_t a = count_smem(E + R), b = scatter_smem(E + R);
  return a > b ? a : b;
}

cudaError_t prepare_layout_kernels() {
  const int max_smem = static_cast<int>(layout_smem_bytes(MOE_MAX_EXPERTS, MOE_MAX_EXPERTS));
  cudaError_t e = cudaFuncSetAttribute(layout_count_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(layout_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

cudaError_t launch_layout(const moe_handle* h, const int32_t* idx, int T, cudaStream_t s) {
  const moe_config& c = h->cfg;
  LayoutArgs a;
  a.idx = idx;
  a.T = T;
  a.K = c.top_k;
  a.E = c.num_experts;
  a.R = c.num_ranks;
  a.epr = c.num_experts / c.num_ranks;
  a.ntiles = T > 0 ? (T + kTile - 1) / kTile : 1;
  a.max_tiles = h->max_tiles;
  a.flags = h->flags;
  a.ticket = h->ticket;
  a.cnt_e = h->cnt_e;
  a.off_e = h->off_e;
  a.cnt_send_r = h->cnt_send_r;
  a.off_send_r = h->off_send_r;
  a.cnt_recv_r = h->cnt_recv_r;
  a.off_recv_r = h->off_recv_r;
  a.S = h->S;
  a.pos = h->pos;
  a.recv_token = h->recv_token;
  a.recv_k = h->recv_k;
  a.send_token = h->send_token;
  a.send_row_of = h->send_row_of;
  a.recv_send_row = h->recv_send_row;
  a.tile_hist = h->tile_hist;

  const int cols = a.E + a.R;
  layout_count_kernel<<<a.ntiles, kThreads, count_smem(cols), s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  layout_scatter_kernel<<<a.ntiles, kThreads, scatter_smem(cols), s>>>(a);
  return cudaGetLastError();
}

int layout_tiles(int T) { return T > 0 ? (T + kTile - 1) / kTile : 1; }

// The same two launches as launch_layout, over caller-chosen buffers: the
// outputs in `out`, the status word `flags` (may be null), and the scratch
// (arrival ticket, zero on entry, and max_tiles * (E + R) tile counters).
cudaError_t launch_layout_buffers(const moe_config& c, const int32_t* idx, int T,
                                  const moe_layout& out, uint32_t* flags, uint32_t* ticket,
                                  int32_t* tile_hist, int max_tiles, cudaStream_t s) {
  LayoutArgs a;
  a.idx = idx;
  a.T = T;
  a.K = c.top_k;
  a.E = c.num_experts;
  a.R = c.num_ranks;
  a.epr = c.num_experts / c.num_ranks;
  a.ntiles = layout_tiles(T);
  a.max_tiles = max_tiles;
  a.flags = flags;
  a.ticket = ticket;
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
  layout_count_kernel<<<a.ntiles, kThreads, count_smem(cols), s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  layout_scatter_kernel<<<a.ntiles, kThreads, scatter_smem(cols), s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
