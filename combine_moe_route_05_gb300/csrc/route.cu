// Top-K routing, one warp per token (sm_103a).
//
// Softmax routing selects the K largest logits (softmax is strictly
// increasing, so the set and order equal those of the probabilities) and
// weights them by softmax; group-limited sigmoid routing selects on
// key = sigmoid(logit) + score-correction bias and weights by the unbiased
// sigmoid (DeepSpeed "Avoid collective token preparation for AutoEP DeepEP",
// "Testing Done": exact routes, score-correction bias).  Selection order is
// descending key, equal keys to the lower expert index.  Weights are computed
// in fp64 and rounded once to fp32.
//
// The sigmoid selection is defined on fp64 keys, but fp64 arithmetic is slow
// on this GPU, so the kernel first selects on fp32 keys and keeps that result
// only when it provably equals the fp64 one:
//   |key32 - key64| <= DELTA = 5e-7 + 1.25e-7 * max|key32| for every expert
// (expf is accurate to 2 ulp, i.e. 2^-22 relative; 1 + e and the reciprocal
// are each rounded once, 2^-24; so the sigmoid is within 1.5 * 2^-22 of its
// value, at most 3.6e-7 since it is <= 1; adding the bias rounds once more,
// 2^-24 |key|; fp64 keys are exact to 1e-15).  A group score (sum of the
// group's top GK keys) is then within GK * (DELTA + 1.25e-7 * max|gs|) of the
// fp64 one, since a top-m sum moves by at most m times the largest change of
// its inputs.  If the fp32 gap between the last kept and the first dropped
// group exceeds twice that bound, and the gap between each of the K + 1 best
// eligible experts and the next exceeds 2 * DELTA, the fp64 selection is the
// same set in the same order; otherwise the token is recomputed in fp64.
//
// Each lane holds VPL consecutive experts (e = lane*VPL + j).  The fp64
// weights of the K selected experts of TB = 32 / K tokens are computed
// together, one (token, k) per lane, so each fp64 instruction serves TB
// tokens.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // warps per block
constexpr unsigned kFull = 0xffffffffu;
constexpr float kDeltaAbs = 5e-7f;
constexpr float kDeltaRel = 1.25e-7f;

struct RouteArgs {
  const float* logits;
  const float* bias;
  int T, E, K;
  int G, TG, GK;
  int renorm;
  int vec4;
  int fast;  // the fp32 selection applies to this configuration
  double scale;
  int32_t* idx;
  float* w;
  uint32_t* flags;
};

template <typename V>
__device__ __forceinline__ bool ranks_before(V kv, int e, V bv, int bi) {
  return kv > bv || (kv == bv && e < bi);
}

// (kv, e) comes strictly after (pv, pi) in the order key desc, index asc.
template <typename V>
__device__ __forceinline__ bool comes_after(V kv, int e, V pv, int pi) {
  return kv < pv || (kv == pv && e > pi);
}

template <typename V>
__device__ __forceinline__ void warp_best(V& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    V ov = __shfl_xor_sync(kFull, v, off);
    int oi = __shfl_xor_sync(kFull, i, off);
    if (ranks_before(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// fp32 -> uint32 with the same order (for -inf..+inf; no NaN reaches here)
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Loads the lane's VPL logits of row t; entries past E read as -inf, NaN as
// -inf (flagged with the other non-finite values).
template <int VPL>
__device__ __forceinline__ bool load_logits(const RouteArgs& a, int t, int lane, float (&v)[VPL]) {
  const float* row = a.logits + static_cast<size_t>(t) * a.E;
  bool bad = false;
  if (VPL >= 4 && a.vec4) {
#pragma unroll
    for (int j = 0; j < VPL; j += 4) {
      const int e = lane * VPL + j;
      float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e < a.E) f = __ldg(reinterpret_cast<const float4*>(row + e));
      v[j] = f.x;
      if (j + 1 < VPL) v[j + 1] = f.y;
      if (j + 2 < VPL) v[j + 2] = f.z;
      if (j + 3 < VPL) v[j + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane * VPL + j;
      v[j] = e < a.E ? __ldg(row + e) : -INFINITY;
    }
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane * VPL + j;
    if (e < a.E && !isfinite(v[j])) {
      bad = true;
      if (isnan(v[j])) v[j] = -INFINITY;
    }
  }
  return bad;
}

// ---------------------------------------------------------------------------
// reference-precision paths, one token at a time (all lanes take part)

// Sigmoid routing of token t entirely in fp64 (keys, group scores,
// selection and weights); writes idx and w.  wkeys: E doubles of shared
// memory owned by this warp.
template <int VPL>
__device__ void sigmoid_token_fp64(const RouteArgs& a, int t, int lane, const float (&v)[VPL],
                                   double* wkeys) {
  const int gsz = a.E / a.G;
  double s[VPL], key[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane * VPL + j;
    if (e < a.E) {
      s[j] = 1.0 / (1.0 + exp(-static_cast<double>(v[j])));
      key[j] = s[j] + (a.bias ? static_cast<double>(__ldg(a.bias + e)) : 0.0);
    } else {
      s[j] = 0.0;
      key[j] = -INFINITY;
    }
  }
  uint32_t keep = 0xffffffffu;
  if (a.G > 1) {
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (lane * VPL + j < a.E) wkeys[lane * VPL + j] = key[j];
    __syncwarp();
    double gscore = -INFINITY;
    if (lane < a.G) {
      const int base = lane * gsz;
      double sum = 0.0, qv = INFINITY;
      int qi = -1;
      for (int r = 0; r < a.GK; ++r) {
        double bv = -INFINITY;
        int bi = INT_MAX;
        for (int i = 0; i < gsz; ++i) {
          const double kv = wkeys[base + i];
          if (comes_after(kv, base + i, qv, qi) && ranks_before(kv, base + i, bv, bi)) {
            bv = kv;
            bi = base + i;
          }
        }
        sum += bv;
        qv = bv;
        qi = bi;
      }
      gscore = sum;
    }
    __syncwarp();
    keep = 0;
    double pv = INFINITY;
    int pi = -1;
    for (int r = 0; r < a.TG; ++r) {
      double bv = -INFINITY;
      int bi = INT_MAX;
      if (lane < a.G && comes_after(gscore, lane, pv, pi)) {
        bv = gscore;
        bi = lane;
      }
      warp_best(bv, bi);
      if (bi < 32) keep |= 1u << bi;
      pv = bv;
      pi = bi;
    }
  }
  double pv = INFINITY, mys = 0.0;
  int pi = -1, myi = 0;
  for (int k = 0; k < a.K; ++k) {
    double bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane * VPL + j;
      const bool eligible = e < a.E && ((keep >> (e / gsz)) & 1u);
      if (eligible && comes_after(key[j], e, pv, pi) && ranks_before(key[j], e, bv, bi)) {
        bv = key[j];
        bi = e;
      }
    }
    warp_best(bv, bi);
    pv = bv;
    pi = bi;
    double sv = 0.0;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (lane * VPL + j == bi) sv = s[j];
    sv = __shfl_sync(kFull, sv, bi / VPL);
    if (lane == k) {
      mys = sv;
      myi = bi;
    }
  }
  double den = 0.0;
  for (int k = 0; k < a.K; ++k) den += __shfl_sync(kFull, mys, k);
  if (lane < a.K) {
    const double p = a.renorm ? mys / den : mys;
    a.idx[static_cast<size_t>(t) * a.K + lane] = myi;
    a.w[static_cast<size_t>(t) * a.K + lane] = static_cast<float>(p * a.scale);
  }
}

// Softmax routing of token t without renormalisation (the denominator runs
// over all E experts); writes idx and w.
template <int VPL>
__device__ void softmax_token_full(const RouteArgs& a, int t, int lane, const float (&v)[VPL]) {
  uint32_t taken = 0;
  float myv = 0.f;
  int myi = 0;
  for (int k = 0; k < a.K; ++k) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane * VPL + j;
      if (!((taken >> j) & 1u) && ranks_before(v[j], e, bv, bi)) {
        bv = v[j];
        bi = e;
      }
    }
    warp_best(bv, bi);
    if (bi / VPL == lane) taken |= 1u << (bi % VPL);
    if (lane == k) {
      myv = bv;
      myi = bi;
    }
  }
  const double lmax = static_cast<double>(__shfl_sync(kFull, myv, 0));
  double part = 0.0;
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    if (lane * VPL + j < a.E) part += exp(static_cast<double>(v[j]) - lmax);
  double den = 0.0;
  for (int l = 0; l < 32; ++l) den += __shfl_sync(kFull, part, l);
  if (lane < a.K) {
    const double ex = exp(static_cast<double>(myv) - lmax);
    a.idx[static_cast<size_t>(t) * a.K + lane] = myi;
    a.w[static_cast<size_t>(t) * a.K + lane] = static_cast<float>((ex / den) * a.scale);
  }
}

// ---------------------------------------------------------------------------
// fp32 selection of one token; returns false if it cannot be trusted (the
// caller then recomputes the token in fp64).  On success, lane base + k holds
// the k-th selected expert.
//
// Each lane first sorts its VPL (key, j) pairs by key, descending, with a
// stable odd-even transposition network (equal keys keep ascending j), so a
// selection round only compares the lanes' heads: the largest head wins,
// equal heads go to the lowest lane, which holds the lower expert indices.

__device__ __forceinline__ float unorder_key(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

template <int VPL>
__device__ __forceinline__ void sort_desc(float (&k)[VPL], int (&j)[VPL]) {
#pragma unroll
  for (int pass = 0; pass < VPL; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < VPL; i += 2) {
      if (k[i] < k[i + 1]) {
        const float tk = k[i];
        k[i] = k[i + 1];
        k[i + 1] = tk;
        const int tj = j[i];
        j[i] = j[i + 1];
        j[i + 1] = tj;
      }
    }
  }
}

// Sum of the top two (or top one) keys of a group whose keys are spread over
// L lanes (each lane's list sorted), merged over lane bits 1..L/2.
__device__ __forceinline__ float group_top2_fp32(float t0, float t1, int gk, int lanes) {
  for (int off = 1; off < lanes; off <<= 1) {
    const float o0 = __shfl_xor_sync(kFull, t0, off);
    const float o1 = __shfl_xor_sync(kFull, t1, off);
    const float n0 = fmaxf(t0, o0);
    const float n1 = fmaxf(fminf(t0, o0), fmaxf(t1, o1));
    t0 = n0;
    t1 = n1;
  }
  return gk >= 2 ? __fadd_rn(__fadd_rn(0.0f, t0), t1) : t0;
}

template <int VPL, bool SIGMOID>
__device__ __forceinline__ bool select_fp32(const RouteArgs& a, int lane, const float (&v)[VPL],
                                            int base, int& my_idx) {
  float sk[VPL];
  int sj[VPL];
  float maxabs = 0.0f;
  int n_valid = 0;  // experts of this lane below E
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane * VPL + j;
    sj[j] = j;
    if (e < a.E) {
      ++n_valid;
      if (SIGMOID) {
        const float s = __frcp_rn(__fadd_rn(1.0f, expf(-v[j])));
        sk[j] = __fadd_rn(s, a.bias ? __ldg(a.bias + e) : 0.0f);
        maxabs = fmaxf(maxabs, fabsf(sk[j]));
      } else {
        sk[j] = v[j];
      }
    } else {
      sk[j] = -INFINITY;
    }
  }
  float delta = 0.0f;
  if (SIGMOID) {
    // non-negative floats order like their bit patterns
    maxabs = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(maxabs)));
    delta = kDeltaAbs + kDeltaRel * maxabs;
    if (!(delta < 1e-3f)) return false;  // huge or non-finite keys
  }
  sort_desc<VPL>(sk, sj);

  // groups (sigmoid only): lanes of a group are contiguous and L = gsz / VPL
  bool eligible_lane = lane * VPL < a.E;
  if (SIGMOID && a.G > 1) {
    const int gsz = a.E / a.G;
    const int L = gsz / VPL;
    const float gs = group_top2_fp32(sk[0], VPL > 1 ? sk[VPL > 1 ? 1 : 0] : -INFINITY, a.GK, L);
    // lane g < G holds group g's score; TG + 1 rounds of warp arg-max, ties
    // to the lower group
    const bool glane = lane < a.G;
    const float my_gs = __shfl_sync(kFull, gs, (lane * L) & 31);
    const float gmax =
        __uint_as_float(__reduce_max_sync(kFull, glane ? __float_as_uint(fabsf(my_gs)) : 0u));
    uint32_t keep = 0;
    float last = 0.0f, next = -INFINITY;
    const int rounds = a.TG < a.G ? a.TG + 1 : a.TG;
    for (int r = 0; r < rounds; ++r) {
      const bool cand = glane && !((keep >> lane) & 1u);
      const uint32_t bits = cand ? order_key(my_gs) : 0u;
      const uint32_t best = __reduce_max_sync(kFull, bits);
      const int wl = __ffs(__ballot_sync(kFull, cand && bits == best)) - 1;
      const float val = unorder_key(best);
      if (r < a.TG) {
        keep |= 1u << wl;
        last = val;
      } else {
        next = val;
      }
    }
    const float dg = a.GK * (delta + kDeltaRel * gmax);
    if (a.TG < a.G && !(last - next > 2.0f * dg)) return false;
    eligible_lane = eligible_lane && ((keep >> ((lane * VPL) / gsz)) & 1u);
  }

  // K (+1 for the gap check) rounds over the lanes' heads
  int consumed = 0;
  float prev = 0.0f;
  const int n_elig = SIGMOID && a.G > 1 ? a.TG * (a.E / a.G) : a.E;
  const int rounds = SIGMOID ? (a.K < n_elig ? a.K + 1 : a.K) : a.K;
  for (int k = 0; k < rounds; ++k) {
    const bool have = eligible_lane && consumed < n_valid;
    const uint32_t bits = have ? order_key(sk[0]) : 0u;
    const uint32_t best = __reduce_max_sync(kFull, bits);
    const int wl = __ffs(__ballot_sync(kFull, have && bits == best)) - 1;
    const int wj = __shfl_sync(kFull, sj[0], wl & 31);
    const float wv = unorder_key(best);
    if (lane == wl) {
#pragma unroll
      for (int i = 0; i + 1 < VPL; ++i) {
        sk[i] = sk[i + 1];
        sj[i] = sj[i + 1];
      }
      sk[VPL - 1] = -INFINITY;
      ++consumed;
    }
    if (SIGMOID && k > 0 && !(prev - wv > 2.0f * delta)) return false;
    prev = wv;
    if (k < a.K && lane == base + k) my_idx = wl * VPL + wj;
  }
  return true;
}

template <int VPL, bool SIGMOID>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteArgs a) {
  extern __shared__ double route_smem[];
  double* wkeys = route_smem + (threadIdx.x >> 5) * a.E;
  const int lane = threadIdx.x & 31;
  const int TB = 32 / a.K;  // tokens per fp64 weight pass
  const int nwarps = gridDim.x * kRouteWarps;
  const int j_of_lane = lane / a.K, k_of_lane = lane % a.K;
  for (int t0 = (blockIdx.x * kRouteWarps + (threadIdx.x >> 5)) * TB; t0 < a.T; t0 += nwarps * TB) {
    int my_idx = 0;
    float my_logit = 0.0f;
    bool my_fast = false;
    for (int j = 0; j < TB; ++j) {
      const int t = t0 + j;
      if (t >= a.T) break;
      float v[VPL];
      const bool bad = load_logits<VPL>(a, t, lane, v);
      if (__any_sync(kFull, bad) && lane == 0) raise_flag(a.flags, MOE_DEVERR_NONFINITE);
      // a softmax selection on fp32 logits is exact even with infinities; a
      // sigmoid token with a non-finite logit goes to the fp64 path
      const bool use_fast = a.fast && !(SIGMOID && __any_sync(kFull, bad));
      int sel_idx = 0;
      const bool ok = use_fast && select_fp32<VPL, SIGMOID>(a, lane, v, j * a.K, sel_idx);
      if (ok) {
        if (j_of_lane == j) {
          my_idx = sel_idx;
          my_logit = __ldg(a.logits + static_cast<size_t>(t) * a.E + sel_idx);
          my_fast = true;
        }
      } else if (SIGMOID) {
        sigmoid_token_fp64<VPL>(a, t, lane, v, wkeys);
      } else {
        softmax_token_full<VPL>(a, t, lane, v);
      }
    }
    // fp64 weights of the tokens selected in fp32: lane = (token j, rank k)
    const int t = t0 + j_of_lane;
    double val;
    if (SIGMOID) {
      val = 1.0 / (1.0 + exp(-static_cast<double>(my_logit)));
    } else {
      const float top = __shfl_sync(kFull, my_logit, (j_of_lane * a.K) & 31);
      val = exp(static_cast<double>(my_logit) - static_cast<double>(top));
    }
    double den = 0.0;
    for (int k = 0; k < a.K; ++k) den += __shfl_sync(kFull, val, (j_of_lane * a.K + k) & 31);
    if (my_fast && j_of_lane < TB && t < a.T) {
      const double p = (SIGMOID && !a.renorm) ? val : val / den;
      a.idx[static_cast<size_t>(t) * a.K + k_of_lane] = my_idx;
      a.w[static_cast<size_t>(t) * a.K + k_of_lane] = static_cast<float>(p * a.scale);
    }
  }
}

template <int VPL, bool SIGMOID>
void launch_one(const RouteArgs& a, int grid, size_t smem, cudaStream_t s) {
  route_kernel<VPL, SIGMOID><<<grid, kRouteWarps * 32, smem, s>>>(a);
}

}  // namespace

cudaError_t launch_route_topk(const moe_handle* h, const float* logits, const float* bias, int T,
                              int32_t* idx, float* w, cudaStream_t s) {
  const moe_config& c = h->cfg;
  RouteArgs a;
  a.logits = logits;
  a.bias = bias;
  a.T = T;
  a.E = c.num_experts;
  a.K = c.top_k;
  a.G = c.num_groups;
  a.TG = c.topk_groups;
  a.GK = c.group_score_topk;
  a.renorm = c.renorm;
  a.vec4 = (c.num_experts % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  a.scale = c.route_scale;
  a.idx = idx;
  a.w = w;
  a.flags = h->flags;
  if (T == 0) return cudaSuccess;

  const int vpl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : a.E <= 256 ? 8 : 16;
  const bool sigmoid = c.score_fn == MOE_SCORE_SIGMOID;
  if (sigmoid) {
    // fp32 pre-selection needs whole lanes per group, a power-of-two lane
    // count per group, and at most 2 keys per group score
    const int gsz = a.E / a.G;
    const int L = gsz / vpl;
    a.fast = a.G == 1 || (gsz % vpl == 0 && L >= 1 && (L & (L - 1)) == 0 && a.GK <= 2);
  } else {
    a.fast = a.renorm;  // without renormalisation the weights need all E exponentials
  }
  const int TB = 32 / a.K;
  const int warps_needed = (T + TB - 1) / TB;
  const int blocks_needed = (warps_needed + kRouteWarps - 1) / kRouteWarps;
  const int cap = h->num_sms * 16;
  const int grid = blocks_needed < cap ? blocks_needed : cap;
  const size_t smem = sigmoid && a.G > 1 ? static_cast<size_t>(kRouteWarps) * a.E * sizeof(double) : 0;
  switch (vpl) {
    case 1: sigmoid ? launch_one<1, true>(a, grid, smem, s) : launch_one<1, false>(a, grid, smem, s); break;
    case 2: sigmoid ? launch_one<2, true>(a, grid, smem, s) : launch_one<2, false>(a, grid, smem, s); break;
    case 4: sigmoid ? launch_one<4, true>(a, grid, smem, s) : launch_one<4, false>(a, grid, smem, s); break;
    case 8: sigmoid ? launch_one<8, true>(a, grid, smem, s) : launch_one<8, false>(a, grid, smem, s); break;
    default: sigmoid ? launch_one<16, true>(a, grid, smem, s) : launch_one<16, false>(a, grid, smem, s); break;
  }
  return cudaGetLastError();
}

}  // namespace moe
