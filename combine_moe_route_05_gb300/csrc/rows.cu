// Row movement kernels of the MoE path (sm_103a): dispatch, combine, their
// backward passes, and the router-score absorption scaling.
//
// dispatch: token-major, one block per token.  Each 16-byte vector of a
//   token row is read from HBM once and stored to the token's K
//   expert-grouped receive rows (and its deduplicated send rows), so a row is
//   never expanded to [T*K,H] by a separate pass (DeepSpeed "Add an opt-in
//   DeepEP transport ...", "Why": tokens are taken before top-k expansion and
//   replicated by the dispatch itself).  Plain vector stores from many warps
//   keep more writes in flight than bulk (TMA) stores from shared memory did
//   for this one-read, K-write pattern.
// combine / dispatch backward: token-major gather of the K rows of a token
//   with 16-byte streaming loads, fp32 accumulation in k order (fused
//   multiply-add for the weighted sum), one rounding to the row dtype.
// combine backward: reads g[t] once and each y row once; writes the K
//   gradient rows and reduces the K router-score gradients <g_t, y[pos]> in
//   a fixed order (deterministic).
#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "router_grad.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// dispatch: one block per token, 16-byte vectors, each row vector read once
// and stored to the token's K receive rows (and its deduplicated send rows)

struct DispatchArgs {
  const uint8_t* x;
  int64_t pf_bytes;  // bytes of x its first pf_blocks blocks pull into L2 (0: none)
  int64_t pf_chunk;  // bytes per such block, a multiple of 16
  int pf_blocks;
  int64_t row_bytes;
  int nvec;
  int T, K;
  const int32_t* pos;
  const float* w;
  const int32_t* send_row_of;
  uint8_t* recv;
  float* recv_w;
  uint8_t* send;
  int recv_rows, send_rows;  // rows of recv / recv_w and of send
  uint32_t* flags;
};

// Pulls bytes [p, p + n) of global memory into L2 (a bulk prefetch; p 16-byte
// aligned, n a multiple of 16), in pieces of 64 KB.  A hint: no data moves
// to the SM and nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, int64_t n) {
  for (int64_t o = 0; o < n; o += 65536) {
    const uint32_t m = static_cast<uint32_t>(n - o < 65536 ? n - o : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + o), "r"(m) : "memory");
  }
}

template <int KMAX, bool kPrefetch>
__global__ void __launch_bounds__(1024) dispatch_kernel(DispatchArgs a) {
  // before the wait for the layout (whose few blocks, and the routing before
  // them, leave HBM nearly idle) the first blocks pull x into L2
  if (kPrefetch && threadIdx.x == 0 && blockIdx.x < a.pf_blocks) {
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * a.pf_chunk;
    const int64_t left = a.pf_bytes - lo;
    if (left > 0) prefetch_l2(a.x + lo, a.pf_chunk < left ? a.pf_chunk : left);
  }
  grid_dependency_wait();
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    int p[KMAX], srow[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      p[k] = -1;
      srow[k] = -1;
      if (k < a.K) {
        p[k] = checked_row(__ldg(a.pos + static_cast<size_t>(t) * a.K + k), a.recv_rows, a.flags);
        if (a.send)
          srow[k] = checked_row(__ldg(a.send_row_of + static_cast<size_t>(t) * a.K + k),
                                a.send_rows, a.flags);
      }
    }
    if (a.send) {
      // a send row is written once, by the lowest k that maps to it
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int j = 0; j < k; ++j)
          if (srow[j] == srow[k]) srow[k] = -1;
    }
    if (a.recv_w && threadIdx.x < a.K) {
      const int pk = __ldg(a.pos + static_cast<size_t>(t) * a.K + threadIdx.x);
      if (static_cast<unsigned>(pk) < static_cast<unsigned>(a.recv_rows))
        a.recv_w[pk] = __ldg(a.w + static_cast<size_t>(t) * a.K + threadIdx.x);
    }
    const uint8_t* xrow = a.x + static_cast<int64_t>(t) * a.row_bytes;
    for (int v = threadIdx.x; v < a.nvec; v += blockDim.x) {
      const Vec16 val = ld_vec(xrow + v * 16);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (p[k] >= 0) st_vec_cs(a.recv + static_cast<int64_t>(p[k]) * a.row_bytes + v * 16, val);
        if (srow[k] >= 0) st_vec_cs(a.send + static_cast<int64_t>(srow[k]) * a.row_bytes + v * 16, val);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// combine / dispatch backward: out[t] = round(sum_k w_k * y[pos[t,k]])

constexpr int kRowThreads = 256;      // elementwise and per-entry kernels
constexpr int kGatherMaxThreads = 512; // combine-type kernels: about 2 vectors per thread

template <typename Elt>
struct RowArgs {
  const uint8_t* y;   // [rows, H] gathered rows
  const uint8_t* g;   // [T, H] (combine backward)
  const float* w;     // [T, K] or NULL
  const int32_t* pos; // [T, K]
  uint8_t* out;       // [T, H] (combine) or [rows, H] (combine backward)
  float* gw;          // [T, K] or NULL
  int64_t row_bytes;
  int nvec;           // 16-byte vectors per row
  int T, K;
  int rows;           // receive rows of y / gy (the bound of every pos entry)
  uint32_t* flags;
  // router backward fused into the dispatch backward (else unused)
  const float* logits;  // [T, E]
  const int32_t* idx;   // [T, K]
  float* glogits;       // [T, E]
  int E;
  int sigmoid, renorm, vec4_e;
  double scale;
};

template <int KMAX>
__device__ __forceinline__ void load_entries(const int32_t* pos, const float* w, int t, int K,
                                             int rows, uint32_t* flags, int (&p)[KMAX],
                                             float (&wk)[KMAX]) {
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    p[k] = -1;
    wk[k] = 1.0f;
    if (k < K) {
      p[k] = checked_row(__ldg(pos + static_cast<size_t>(t) * K + k), rows, flags);
      if (w) wk[k] = __ldg(w + static_cast<size_t>(t) * K + k);
    }
  }
}

// Router backward to the logits for TB = 32/K tokens of this block, its
// tokens j0 .. j0+TB-1 (t = blockIdx.x + j*gridDim.x, j < ntok), by one warp:
// lane jj*K + k takes entry k of token j0 + jj.  The tokens' rows of glogits
// are zeroed, then their K entries written (router_grad_entry: fp64, rounded
// once), from the complete score gradient gw.
template <typename Elt>
__device__ __noinline__ void router_bwd_pass(const RowArgs<Elt>& a, int j0, int ntok) {
  const int lane = threadIdx.x & 31;
  const int TB = 32 / a.K;
  const int jj = lane / a.K, k = lane % a.K;
  for (int u = 0; u < TB && j0 + u < ntok; ++u) {
    float* row = a.glogits + static_cast<size_t>(blockIdx.x + (j0 + u) * gridDim.x) * a.E;
    if (a.vec4_e) {
      for (int e = lane * 4; e < a.E; e += 128)
        *reinterpret_cast<float4*>(row + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      for (int e = lane; e < a.E; e += 32) row[e] = 0.f;
    }
  }
  const int j = j0 + jj;
  const bool valid = jj < TB && j < ntok;
  const int t = blockIdx.x + j * gridDim.x;
  int e = 0;
  double l = 0.0, g = 0.0;
  if (valid) {
    const size_t tk = static_cast<size_t>(t) * a.K + k;
    e = __ldg(a.idx + tk);
    if (e < 0 || e >= a.E) e = 0;  // as the separate router backward
    l = static_cast<double>(__ldg(a.logits + static_cast<size_t>(t) * a.E + e));
    g = static_cast<double>(__ldg(a.gw + tk));
  }
  const double d = router_grad_entry(l, g, (jj * a.K) & 31, a.K, a.sigmoid != 0, a.renorm != 0,
                                     a.scale);
  __syncwarp();  // the zero fill above is ordered before these writes
  if (valid) a.glogits[static_cast<size_t>(t) * a.E + e] = static_cast<float>(d);
}

// combine: out[t] = round(sum_k w_k y[pos[t,k]]) (or the plain sum) in fp32,
// k in order.  ROUTE (the dispatch backward with the router backward fused
// in) also runs the router backward of the block's tokens, TB = 32/K tokens
// per pass, each pass by the next warp in turn before its rows of the pass's
// first token: there is no barrier between the warps, so the fp64 latency of
// a pass hides behind the other warps' row traffic.
template <typename Elt, int KMAX, bool WEIGHTED, bool ROUTE>
__device__ __forceinline__ void combine_body(const RowArgs<Elt>& a) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  int ntok = 0, TB = 1, nw = 1;
  if (ROUTE) {
    ntok = a.T > static_cast<int>(blockIdx.x)
               ? (a.T - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
               : 0;
    TB = 32 / a.K;
    nw = blockDim.x >> 5;
  }
  int it = 0;
  for (int t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
    if (ROUTE && it % TB == 0 && static_cast<int>(threadIdx.x >> 5) == (it / TB) % nw)
      router_bwd_pass(a, it, ntok);
    int p[KMAX];
    float wk[KMAX];
    load_entries<KMAX>(a.pos, WEIGHTED ? a.w : nullptr, t, a.K, a.rows, a.flags, p, wk);
    uint8_t* orow = a.out + static_cast<int64_t>(t) * a.row_bytes;
    for (int v = threadIdx.x; v < a.nvec; v += blockDim.x) {
      Vec16 in[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (p[k] >= 0) in[k] = ld_stream(a.y + static_cast<int64_t>(p[k]) * a.row_bytes + v * 16);
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (p[k] < 0) continue;
        float f[N];
        VT::to_f32(in[k], f);
#pragma unroll
        for (int i = 0; i < N; ++i)
          acc[i] = WEIGHTED ? __fmaf_rn(wk[k], f[i], acc[i]) : __fadd_rn(acc[i], f[i]);
      }
      st_vec(orow + v * 16, VT::from_f32(acc));
    }
  }
}

template <typename Elt, int KMAX, bool WEIGHTED>
__global__ void __launch_bounds__(kGatherMaxThreads) combine_kernel(RowArgs<Elt> a) {
  combine_body<Elt, KMAX, WEIGHTED, false>(a);
}

// the dispatch backward with the router backward fused in: two blocks per SM
// (the row loop's occupancy), the router pass out of line
template <typename Elt, int KMAX>
__global__ void __launch_bounds__(kGatherMaxThreads, 2) dispatch_bwd_route_kernel(RowArgs<Elt> a) {
  combine_body<Elt, KMAX, false, true>(a);
}

// One token of the combine backward for the row threads tid = 0 .. nthr-1 of
// the block: gy[pos[t,k]] = round(w_k * g[t]) (or g[t]) for its 16-byte
// vectors v = tid, tid + nthr, ..., and (DOT) its fp32 partial dot products
// <g[t], y[pos[t,k]]> over those vectors, reduced across the warp.
template <typename Elt, int KMAX, bool WEIGHTED, bool DOT>
__device__ __forceinline__ void combine_bwd_token(const RowArgs<Elt>& a, int t, int tid, int nthr,
                                                  float (&dot)[KMAX]) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  int p[KMAX];
  float wk[KMAX];
  load_entries<KMAX>(a.pos, WEIGHTED ? a.w : nullptr, t, a.K, a.rows, a.flags, p, wk);
#pragma unroll
  for (int k = 0; k < KMAX; ++k) dot[k] = 0.0f;
  const uint8_t* grow = a.g + static_cast<int64_t>(t) * a.row_bytes;
  for (int v = tid; v < a.nvec; v += nthr) {
    const Vec16 gv = ld_stream(grow + v * 16);
    Vec16 yv[KMAX];
    if (DOT) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (p[k] >= 0) yv[k] = ld_vec(a.y + static_cast<int64_t>(p[k]) * a.row_bytes + v * 16);
    }
    float gf[N];
    VT::to_f32(gv, gf);
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (p[k] < 0) continue;
      uint8_t* dst = a.out + static_cast<int64_t>(p[k]) * a.row_bytes + v * 16;
      if (WEIGHTED) {
        float o[N];
#pragma unroll
        for (int i = 0; i < N; ++i) o[i] = __fmul_rn(wk[k], gf[i]);
        st_vec(dst, VT::from_f32(o));
      } else {
        st_vec(dst, gv);
      }
      if (DOT) {
        float yf[N];
        VT::to_f32(yv[k], yf);
#pragma unroll
        for (int i = 0; i < N; ++i) dot[k] = __fmaf_rn(gf[i], yf[i], dot[k]);
      }
    }
  }
  if (DOT) {
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot[k] += __shfl_xor_sync(kFull, dot[k], off);
    }
  }
}

// combine backward: gy[pos[t,k]] = round(w_k * g[t]) (or g[t]), and
// gw[t,k] = <g[t], y[pos[t,k]]> reduced over the block in a fixed order
// (warp partials summed in warp order).
template <typename Elt, int KMAX, bool WEIGHTED, bool DOT>
__global__ void __launch_bounds__(kGatherMaxThreads, 2) combine_bwd_kernel(RowArgs<Elt> a) {
  __shared__ float red[2][kGatherMaxThreads / 32][KMAX];
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int it = 0;
  for (int t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
    float dot[KMAX];
    combine_bwd_token<Elt, KMAX, WEIGHTED, DOT>(a, t, threadIdx.x, blockDim.x, dot);
    if (DOT) {
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < KMAX; ++k) red[it & 1][warp][k] = dot[k];
      }
      __syncthreads();
      if (threadIdx.x < a.K) {
        float s = 0.0f;
        for (int wi = 0; wi < nw; ++wi) s += red[it & 1][wi][threadIdx.x];
        const int pk = __ldg(a.pos + static_cast<size_t>(t) * a.K + threadIdx.x);
        a.gw[static_cast<size_t>(t) * a.K + threadIdx.x] =
            static_cast<unsigned>(pk) < static_cast<unsigned>(a.rows) ? s : 0.0f;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// pad rows of a padded receive layout: zeros (one block per expert)

__global__ void __launch_bounds__(256) zero_pad_rows_kernel(uint8_t* rows, int64_t row_bytes,
                                                            const int32_t* off_e,
                                                            const int32_t* cnt_e, int E,
                                                            int nrows, uint32_t* flags) {
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    int64_t lo = static_cast<int64_t>(off_e[e]) + cnt_e[e], hi = off_e[e + 1];
    if (lo < 0 || hi > nrows) {
      // offsets outside the tensor: zero only what lies inside it
      if (threadIdx.x == 0) raise_flag(flags, MOE_DEVERR_BAD_LAYOUT);
      lo = lo < 0 ? 0 : lo;
      hi = hi > nrows ? nrows : hi;
    }
    uint8_t* base = rows + lo * row_bytes;
    const int64_t bytes = (hi - lo) * row_bytes;
    if ((row_bytes & 15) == 0) {
      const Vec16 z{{0u, 0u, 0u, 0u}};
      for (int64_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) st_vec(base + i * 16, z);
    } else {
      for (int64_t i = threadIdx.x; i < bytes / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(base)[i] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// staged (wire-faithful) mode: a token's row goes to each destination rank
// once (its send row); the receiving side expands it to the rows of its
// experts there, and the combine returns one partial row per send row, which
// the token's side then adds up.  One block per token; a send row's entries
// are the k with equal send_row_of, handled from the first such k.

struct StagedArgs {
  const uint8_t* src;  // send rows (expand), y (partial), partial rows (reduce)
  const float* w;
  const int32_t* pos;
  const int32_t* send_row_of;
  uint8_t* dst;        // recv (expand), partial (partial), out (reduce)
  int64_t row_bytes;
  int nvec;
  int T, K;
  int recv_rows, send_rows;  // bounds of pos and send_row_of entries
  uint32_t* flags;
};

template <int KMAX>
__device__ __forceinline__ uint32_t load_send_entries(const StagedArgs& a, int t, int (&p)[KMAX],
                                                      int (&sr)[KMAX]) {
  uint32_t first = 0;  // bit k: first entry of its send row
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    p[k] = -1;
    sr[k] = -1;
    if (k < a.K) {
      p[k] = checked_row(__ldg(a.pos + static_cast<size_t>(t) * a.K + k), a.recv_rows, a.flags);
      sr[k] = checked_row(__ldg(a.send_row_of + static_cast<size_t>(t) * a.K + k), a.send_rows,
                          a.flags);
    }
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    bool f = sr[k] >= 0;
#pragma unroll
    for (int j = 0; j < k; ++j)
      if (sr[j] == sr[k]) f = false;
    if (f) first |= 1u << k;
  }
  return first;
}

// recv[pos[t,k]] = send[send_row_of[t,k]]: each send row read once
template <int KMAX>
__global__ void __launch_bounds__(kGatherMaxThreads) expand_kernel(StagedArgs a) {
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    int p[KMAX], sr[KMAX];
    const uint32_t first = load_send_entries<KMAX>(a, t, p, sr);
    for (int v = threadIdx.x; v < a.nvec; v += blockDim.x) {
      // all of the token's send-row loads first, so they are in flight
      // together (the loads and stores are ordered asm statements)
      Vec16 val[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if ((first >> k) & 1u)
          val[k] = ld_stream(a.src + static_cast<int64_t>(sr[k]) * a.row_bytes + v * 16);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (!((first >> k) & 1u)) continue;
#pragma unroll
        for (int j = k; j < KMAX; ++j)
          if (sr[j] == sr[k] && p[j] >= 0)
            st_vec(a.dst + static_cast<int64_t>(p[j]) * a.row_bytes + v * 16, val[k]);
      }
    }
  }
}

// partial[s] = round(sum over the entries of send row s, in k order, of
// w_k * y[pos[t,k]])
template <typename Elt, int KMAX, bool WEIGHTED>
__global__ void __launch_bounds__(kGatherMaxThreads) combine_partial_kernel(StagedArgs a) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    int p[KMAX], sr[KMAX];
    const uint32_t first = load_send_entries<KMAX>(a, t, p, sr);
    float wk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      wk[k] = (WEIGHTED && k < a.K) ? __ldg(a.w + static_cast<size_t>(t) * a.K + k) : 1.0f;
    for (int v = threadIdx.x; v < a.nvec; v += blockDim.x) {
      Vec16 in[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (p[k] >= 0) in[k] = ld_stream(a.src + static_cast<int64_t>(p[k]) * a.row_bytes + v * 16);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (!((first >> k) & 1u)) continue;
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = k; j < KMAX; ++j) {
          if (sr[j] != sr[k] || p[j] < 0) continue;
          float f[N];
          VT::to_f32(in[j], f);
#pragma unroll
          for (int i = 0; i < N; ++i)
            acc[i] = WEIGHTED ? __fmaf_rn(wk[j], f[i], acc[i]) : __fadd_rn(acc[i], f[i]);
        }
        st_vec(a.dst + static_cast<int64_t>(sr[k]) * a.row_bytes + v * 16, VT::from_f32(acc));
      }
    }
  }
}

// out[t] = round(sum of the token's partial rows, each send row once, in the
// order of its first entry)
template <typename Elt, int KMAX>
__global__ void __launch_bounds__(kGatherMaxThreads) combine_reduce_kernel(StagedArgs a) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    int p[KMAX], sr[KMAX];
    const uint32_t first = load_send_entries<KMAX>(a, t, p, sr);
    for (int v = threadIdx.x; v < a.nvec; v += blockDim.x) {
      Vec16 in[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if ((first >> k) & 1u)
          in[k] = ld_stream(a.src + static_cast<int64_t>(sr[k]) * a.row_bytes + v * 16);
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (!((first >> k) & 1u)) continue;
        float f[N];
        VT::to_f32(in[k], f);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
      }
      st_vec(a.dst + static_cast<int64_t>(t) * a.row_bytes + v * 16, VT::from_f32(acc));
    }
  }
}

// ---------------------------------------------------------------------------
// absorption: hs[r] = round(h[r] * recv_w[r]) over the valid receive rows

template <typename Elt>
__global__ void __launch_bounds__(kRowThreads) scale_rows_kernel(const uint8_t* h, const float* rw,
                                                                 uint8_t* hs, int64_t row_bytes,
                                                                 int nvec, const int32_t* nrows_dev,
                                                                 int rows_cap, uint32_t* flags) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  int64_t nrows = *nrows_dev;
  if (nrows < 0 || nrows > rows_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_flag(flags, MOE_DEVERR_BAD_LAYOUT);
    nrows = nrows < 0 ? 0 : rows_cap;
  }
  const int64_t total = nrows * nvec;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kRowThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kRowThreads) {
    const int64_t r = i / nvec;
    const int v = static_cast<int>(i - r * nvec);
    const float s = __ldg(rw + r);
    float f[N];
    VT::to_f32(ld_stream(h + r * row_bytes + v * 16), f);
#pragma unroll
    for (int j = 0; j < N; ++j) f[j] = __fmul_rn(f[j], s);
    st_vec(hs + r * row_bytes + v * 16, VT::from_f32(f));
  }
}

// absorption backward, one warp per entry (t,k):
//   gh[p] = round(recv_w[p] * ghs[p]),  gw[t,k] = <ghs[p], h[p]>,  p = pos[t,k]
template <typename Elt>
__global__ void __launch_bounds__(kRowThreads) scale_rows_bwd_kernel(
    const uint8_t* ghs, const uint8_t* h, const float* rw, uint8_t* gh, float* gw,
    const int32_t* pos, int64_t entries, int64_t row_bytes, int nvec, int rows,
    uint32_t* flags) {
  using VT = VecTraits<Elt>;
  constexpr int N = VT::N;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kRowThreads / 32);
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5);
       e < entries; e += nwarps) {
    const int p = checked_row(__ldg(pos + e), rows, flags);
    float dot = 0.0f;
    if (p >= 0) {
      const float s = __ldg(rw + p);
      const uint8_t* grow = ghs + static_cast<int64_t>(p) * row_bytes;
      const uint8_t* hrow = h + static_cast<int64_t>(p) * row_bytes;
      uint8_t* orow = gh + static_cast<int64_t>(p) * row_bytes;
      for (int v = lane; v < nvec; v += 32) {
        float gf[N], hf[N], o[N];
        VT::to_f32(ld_vec(grow + v * 16), gf);
        VT::to_f32(ld_vec(hrow + v * 16), hf);
#pragma unroll
        for (int j = 0; j < N; ++j) {
          o[j] = __fmul_rn(s, gf[j]);
          dot = __fmaf_rn(gf[j], hf[j], dot);
        }
        st_vec(orow + v * 16, VT::from_f32(o));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
    }
    if (lane == 0) gw[e] = dot;
  }
}

// Threads per block for rows of nvec 16-byte vectors, `per` vectors per
// thread: whole warps, at most 1024.
int threads_for(int nvec, int per) {
  int t = (nvec + per - 1) / per;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > 1024 ? 1024 : t);
}

}  // namespace

// Resident blocks per SM of `kernel`, computed once per (kernel, smem) pair.
int resident_blocks(const void* kernel, int threads, size_t smem) {
  struct Entry {
    const void* k;
    int threads;
    size_t smem;
    int per_sm;
  };
  static Entry cache[32];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].k == kernel && cache[i].threads == threads && cache[i].smem == smem)
      return cache[i].per_sm;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
    per_sm = 1;
  if (per_sm < 1) per_sm = 1;
  if (used < 32) cache[used++] = Entry{kernel, threads, smem, per_sm};
  return per_sm;
}

namespace {

// Persistent grid: every resident block slot of the GPU, or fewer if there is
// less work.
int grid_for(const void* kernel, int threads, size_t smem, int num_sms, long long work_items) {
  long long g = static_cast<long long>(resident_blocks(kernel, threads, smem)) * num_sms;
  if (work_items < g) g = work_items;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Rows of a receive-row tensor (T*K plus the pads) and of a send-row tensor
// (T*min(K,R)) for the handle's current layout: the bounds of the layout's
// row indices.
int recv_rows_of(const moe_handle* h) {
  return h->T * h->cfg.top_k + h->cfg.num_experts * (h->pad - 1);
}
int send_rows_of(const moe_handle* h) {
  return h->T * (h->cfg.top_k < h->cfg.num_ranks ? h->cfg.top_k : h->cfg.num_ranks);
}

int gather_threads(int nvec) {
  const int t = threads_for(nvec, 2);
  return t > kGatherMaxThreads ? kGatherMaxThreads : t;
}

template <typename Elt, int KMAX>
cudaError_t launch_combine_t(const moe_handle* h, const void* y, int H, const float* w, void* out,
                             cudaStream_t s, const RouterBwdRows* rt = nullptr) {
  RowArgs<Elt> a{};
  a.y = static_cast<const uint8_t*>(y);
  a.w = w;
  a.pos = h->pos;
  a.out = static_cast<uint8_t*>(out);
  a.row_bytes = static_cast<int64_t>(H) * sizeof(Elt);
  a.nvec = static_cast<int>(a.row_bytes / 16);
  a.T = h->T;
  a.K = h->cfg.top_k;
  a.rows = recv_rows_of(h);
  a.flags = h->flags;
  if (a.T == 0) return cudaSuccess;
  const int block = gather_threads(a.nvec);
  if (rt) {
    a.logits = rt->logits;
    a.idx = rt->idx;
    a.gw = const_cast<float*>(rt->gw);
    a.glogits = rt->glogits;
    a.E = h->cfg.num_experts;
    a.sigmoid = h->cfg.score_fn == MOE_SCORE_SIGMOID;
    a.renorm = h->cfg.renorm;
    a.scale = h->cfg.route_scale;
    a.vec4_e = (a.E % 4) == 0 && (reinterpret_cast<uintptr_t>(rt->glogits) & 15) == 0;
    auto k = dispatch_bwd_route_kernel<Elt, KMAX>;
    k<<<grid_for(reinterpret_cast<const void*>(k), block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  } else if (w) {
    auto k = combine_kernel<Elt, KMAX, true>;
    k<<<grid_for(reinterpret_cast<const void*>(k), block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  } else {
    auto k = combine_kernel<Elt, KMAX, false>;
    k<<<grid_for(reinterpret_cast<const void*>(k), block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  }
  return cudaGetLastError();
}

template <typename Elt, int KMAX>
cudaError_t launch_combine_bwd_t(const moe_handle* h, const void* g, const void* y, int H,
                                 const float* w, void* gy, float* gw, cudaStream_t s) {
  RowArgs<Elt> a{};
  a.y = static_cast<const uint8_t*>(y);
  a.g = static_cast<const uint8_t*>(g);
  a.w = w;
  a.pos = h->pos;
  a.out = static_cast<uint8_t*>(gy);
  a.gw = gw;
  a.row_bytes = static_cast<int64_t>(H) * sizeof(Elt);
  a.nvec = static_cast<int>(a.row_bytes / 16);
  a.T = h->T;
  a.K = h->cfg.top_k;
  a.rows = recv_rows_of(h);
  a.flags = h->flags;
  if (a.T == 0) return cudaSuccess;
  // rows of at most 256 vectors (H <= 2048 bf16) take a thread per vector:
  // Qwen3-30B step 255.3 -> 251.0 us; at 512 vectors two per thread stays
  // faster (Qwen3-235B step 2143.7 against 2148 us)
  const int block = a.nvec <= 256 ? threads_for(a.nvec, 1) : gather_threads(a.nvec);
  const void* kp;
  if (w && gw) {
    auto k = combine_bwd_kernel<Elt, KMAX, true, true>;
    kp = reinterpret_cast<const void*>(k);
    k<<<grid_for(kp, block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  } else if (w) {
    auto k = combine_bwd_kernel<Elt, KMAX, true, false>;
    kp = reinterpret_cast<const void*>(k);
    k<<<grid_for(kp, block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  } else {
    auto k = combine_bwd_kernel<Elt, KMAX, false, false>;
    kp = reinterpret_cast<const void*>(k);
    k<<<grid_for(kp, block, 0, h->num_sms, a.T), block, 0, s>>>(a);
  }
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : zero_pad_rows(h, gy, a.row_bytes, s);
}

}  // namespace


cudaError_t launch_dispatch(const moe_handle* h, const void* x, int64_t row_bytes, const float* w,
                            void* recv, float* recv_w, void* send, cudaStream_t s) {
  DispatchArgs a{};
  a.x = static_cast<const uint8_t*>(x);
  a.row_bytes = row_bytes;
  a.nvec = static_cast<int>(row_bytes / 16);
  a.T = h->T;
  a.K = h->cfg.top_k;
  a.pos = h->pos;
  a.w = w;
  a.send_row_of = h->send_row_of;
  a.recv = static_cast<uint8_t*>(recv);
  a.recv_w = recv_w;
  a.send = static_cast<uint8_t*>(send);
  a.recv_rows = recv_rows_of(h);
  a.send_rows = send_rows_of(h);
  a.flags = h->flags;
  if (a.T == 0) return cudaSuccess;
  // one block per token, a thread per 16-byte vector of the row (many
  // independent stores in flight; measured faster than bulk copies through
  // shared memory for this 1-read / K-write pattern)
  const int block = threads_for(a.nvec, 1);
  const int grid = a.T < 1048576 ? a.T : 1048576;
  // x is prefetched into L2 while the layout runs where all of it fits in
  // half the L2 (Qwen3-30B shape, 34 MB: step 251.4 -> 249.0 us); a leading
  // part of a larger x measured slower (DeepSeek-V3, 235 MB: +2 to +10 us
  // for 32 to 96 MB), so there nothing is prefetched
  const int64_t x_bytes = static_cast<int64_t>(a.T) * row_bytes;
  if (x_bytes <= h->l2_bytes / 2) {
    a.pf_bytes = x_bytes;
    a.pf_blocks = grid < 128 ? grid : 128;
    a.pf_chunk = ((x_bytes + a.pf_blocks - 1) / a.pf_blocks + 15) / 16 * 16;
  }
  // chained to the layout before it (its blocks are scheduled while the
  // layout's few blocks run); the row kernels after it are launched plainly,
  // which measured faster than chaining them
  const bool pf = a.pf_bytes > 0;
  if (a.K <= 8)
    (void)launch_chained(pf ? dispatch_kernel<8, true> : dispatch_kernel<8, false>, dim3(grid),
                         dim3(block), 0, s, false, a);
  else
    (void)launch_chained(pf ? dispatch_kernel<16, true> : dispatch_kernel<16, false>, dim3(grid),
                         dim3(block), 0, s, false, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = zero_pad_rows(h, recv, row_bytes, s);
  if (e != cudaSuccess) return e;
  return zero_pad_rows(h, recv_w, sizeof(float), s);
}

cudaError_t launch_combine(const moe_handle* h, const void* y, int H, int dtype, const float* w,
                           void* out, cudaStream_t s) {
  const bool k8 = h->cfg.top_k <= 8;
  if (dtype == MOE_BF16)
    return k8 ? launch_combine_t<__nv_bfloat16, 8>(h, y, H, w, out, s)
              : launch_combine_t<__nv_bfloat16, 16>(h, y, H, w, out, s);
  return k8 ? launch_combine_t<float, 8>(h, y, H, w, out, s)
            : launch_combine_t<float, 16>(h, y, H, w, out, s);
}

cudaError_t launch_combine_bwd(const moe_handle* h, const void* g, const void* y, int H, int dtype,
                               const float* w, void* gy, float* gw, cudaStream_t s) {
  const bool k8 = h->cfg.top_k <= 8;
  if (dtype == MOE_BF16)
    return k8 ? launch_combine_bwd_t<__nv_bfloat16, 8>(h, g, y, H, w, gy, gw, s)
              : launch_combine_bwd_t<__nv_bfloat16, 16>(h, g, y, H, w, gy, gw, s);
  return k8 ? launch_combine_bwd_t<float, 8>(h, g, y, H, w, gy, gw, s)
            : launch_combine_bwd_t<float, 16>(h, g, y, H, w, gy, gw, s);
}

int dispatch_bwd_route_launches(const moe_config& c) {
  return c.score_fn == MOE_SCORE_SOFTMAX && !c.renorm ? 2 : 1;
}

cudaError_t launch_dispatch_bwd_route(const moe_handle* h, const void* grecv, int H, int dtype,
                                      const float* logits, const int32_t* idx, const float* gw,
                                      void* gx, float* glogits, cudaStream_t s) {
  if (dispatch_bwd_route_launches(h->cfg) == 2) {
    const cudaError_t e = launch_combine(h, grecv, H, dtype, nullptr, gx, s);
    return e != cudaSuccess ? e : launch_route_bwd(h, logits, idx, gw, h->T, glogits, s);
  }
  const RouterBwdRows rt{logits, idx, gw, glogits};
  const bool k8 = h->cfg.top_k <= 8;
  if (dtype == MOE_BF16)
    return k8 ? launch_combine_t<__nv_bfloat16, 8>(h, grecv, H, nullptr, gx, s, &rt)
              : launch_combine_t<__nv_bfloat16, 16>(h, grecv, H, nullptr, gx, s, &rt);
  return k8 ? launch_combine_t<float, 8>(h, grecv, H, nullptr, gx, s, &rt)
            : launch_combine_t<float, 16>(h, grecv, H, nullptr, gx, s, &rt);
}

cudaError_t launch_scale_rows(const moe_handle* h, const void* hrows, int I, int dtype,
                              const float* recv_w, void* hs, cudaStream_t s) {
  const int64_t row_bytes = static_cast<int64_t>(I) * (dtype == MOE_BF16 ? 2 : 4);
  const int nvec = static_cast<int>(row_bytes / 16);
  if (h->T == 0) return cudaSuccess;
  const long long items = static_cast<long long>(h->T) * h->cfg.top_k * nvec;
  const long long blocks = (items + kRowThreads - 1) / kRowThreads;
  const int32_t* nrows = h->off_e + h->cfg.num_experts;
  if (dtype == MOE_BF16) {
    auto k = scale_rows_kernel<__nv_bfloat16>;
    const int grid = grid_for(reinterpret_cast<const void*>(k), kRowThreads, 0, h->num_sms, blocks);
    k<<<grid, kRowThreads, 0, s>>>(static_cast<const uint8_t*>(hrows), recv_w,
                                   static_cast<uint8_t*>(hs), row_bytes, nvec, nrows,
                                   recv_rows_of(h), h->flags);
  } else {
    auto k = scale_rows_kernel<float>;
    const int grid = grid_for(reinterpret_cast<const void*>(k), kRowThreads, 0, h->num_sms, blocks);
    k<<<grid, kRowThreads, 0, s>>>(static_cast<const uint8_t*>(hrows), recv_w,
                                   static_cast<uint8_t*>(hs), row_bytes, nvec, nrows,
                                   recv_rows_of(h), h->flags);
  }
  return cudaGetLastError();
}

cudaError_t launch_scale_rows_bwd(const moe_handle* h, const void* ghs, const void* hrows, int I,
                                  int dtype, const float* recv_w, void* gh, float* gw,
                                  cudaStream_t s) {
  const int64_t row_bytes = static_cast<int64_t>(I) * (dtype == MOE_BF16 ? 2 : 4);
  const int nvec = static_cast<int>(row_bytes / 16);
  const int64_t entries = static_cast<int64_t>(h->T) * h->cfg.top_k;
  if (entries == 0) return cudaSuccess;
  const long long blocks = (entries + kRowThreads / 32 - 1) / (kRowThreads / 32);
  if (dtype == MOE_BF16) {
    auto k = scale_rows_bwd_kernel<__nv_bfloat16>;
    const int grid = grid_for(reinterpret_cast<const void*>(k), kRowThreads, 0, h->num_sms, blocks);
    k<<<grid, kRowThreads, 0, s>>>(static_cast<const uint8_t*>(ghs),
                                   static_cast<const uint8_t*>(hrows), recv_w,
                                   static_cast<uint8_t*>(gh), gw, h->pos, entries, row_bytes, nvec,
                                   recv_rows_of(h), h->flags);
  } else {
    auto k = scale_rows_bwd_kernel<float>;
    const int grid = grid_for(reinterpret_cast<const void*>(k), kRowThreads, 0, h->num_sms, blocks);
    k<<<grid, kRowThreads, 0, s>>>(static_cast<const uint8_t*>(ghs),
                                   static_cast<const uint8_t*>(hrows), recv_w,
                                   static_cast<uint8_t*>(gh), gw, h->pos, entries, row_bytes, nvec,
                                   recv_rows_of(h), h->flags);
  }
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : zero_pad_rows(h, gh, row_bytes, s);
}

cudaError_t launch_staged(int op, const moe_handle* h, const void* src, int H, int dtype,
                          const float* w, void* dst, cudaStream_t s) {
  StagedArgs a{};
  a.src = static_cast<const uint8_t*>(src);
  a.w = w;
  a.pos = h->pos;
  a.send_row_of = h->send_row_of;
  a.dst = static_cast<uint8_t*>(dst);
  a.row_bytes = static_cast<int64_t>(H) * (dtype == MOE_BF16 ? 2 : 4);
  a.nvec = static_cast<int>(a.row_bytes / 16);
  a.T = h->T;
  a.K = h->cfg.top_k;
  a.recv_rows = recv_rows_of(h);
  a.send_rows = send_rows_of(h);
  a.flags = h->flags;
  if (a.T == 0) return cudaSuccess;
  const bool k8 = a.K <= 8;
  if (op == 0) {  // expand: one block per token, about two vectors per thread
    const int block = gather_threads(a.nvec);
    const int grid = a.T < 1048576 ? a.T : 1048576;
    if (k8) expand_kernel<8><<<grid, block, 0, s>>>(a);
    else expand_kernel<16><<<grid, block, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    return e != cudaSuccess ? e : zero_pad_rows(h, dst, a.row_bytes, s);
  }
  const int block = gather_threads(a.nvec);
#define MOE_STAGED_LAUNCH(KERNEL)                                                            \
  do {                                                                                       \
    auto kern = KERNEL;                                                                      \
    kern<<<grid_for(reinterpret_cast<const void*>(kern), block, 0, h->num_sms, a.T), block, 0, \
           s>>>(a);                                                                          \
  } while (0)
  if (op == 1) {
    if (dtype == MOE_BF16) {
      if (k8) { if (w) MOE_STAGED_LAUNCH((combine_partial_kernel<__nv_bfloat16, 8, true>)); else MOE_STAGED_LAUNCH((combine_partial_kernel<__nv_bfloat16, 8, false>)); }
      else { if (w) MOE_STAGED_LAUNCH((combine_partial_kernel<__nv_bfloat16, 16, true>)); else MOE_STAGED_LAUNCH((combine_partial_kernel<__nv_bfloat16, 16, false>)); }
    } else {
      if (k8) { if (w) MOE_STAGED_LAUNCH((combine_partial_kernel<float, 8, true>)); else MOE_STAGED_LAUNCH((combine_partial_kernel<float, 8, false>)); }
      else { if (w) MOE_STAGED_LAUNCH((combine_partial_kernel<float, 16, true>)); else MOE_STAGED_LAUNCH((combine_partial_kernel<float, 16, false>)); }
    }
  } else {
    if (dtype == MOE_BF16) {
      if (k8) MOE_STAGED_LAUNCH((combine_reduce_kernel<__nv_bfloat16, 8>));
      else MOE_STAGED_LAUNCH((combine_reduce_kernel<__nv_bfloat16, 16>));
    } else {
      if (k8) MOE_STAGED_LAUNCH((combine_reduce_kernel<float, 8>));
      else MOE_STAGED_LAUNCH((combine_reduce_kernel<float, 16>));
    }
  }
#undef MOE_STAGED_LAUNCH
  return cudaGetLastError();
}

cudaError_t zero_pad_rows(const moe_handle* h, void* rows, int64_t row_bytes, cudaStream_t s) {
  if (h->pad <= 1 || h->T <= 0 || !rows) return cudaSuccess;
  const int E = h->cfg.num_experts;
  zero_pad_rows_kernel<<<E, 256, 0, s>>>(static_cast<uint8_t*>(rows), row_bytes, h->off_e, h->cnt_e,
                                          E, recv_rows_of(h), h->flags);
  return cudaGetLastError();
}

}  // namespace moe
