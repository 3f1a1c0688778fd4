// Top-K routing (sm_103a): eight threads per token where E is 64, 128 or 256
// and K <= 8 (route_team_kernel), else one warp per token (route_kernel).
//
// Softmax routing selects the K largest logits (softmax is strictly
// increasing, so the set and order equal those of the probabilities) and
// weights them by softmax; group-limited sigmoid routing selects on
// key = sigmoid(logit) + score-correction bias and weights by the unbiased
// sigmoid (DeepSpeed "Avoid collective token preparation for AutoEP DeepEP",
// "Testing Done": exact routes, score-correction bias).  Selection order is
// descending key, equal keys to the lower expert index.  Weights follow the
// fp64 definition (float-float arithmetic below, rounded once to fp32).
//
// The sigmoid selection is defined on fp64 keys, but fp64 arithmetic is slow
// on this GPU, so the kernel first selects on fp32 keys and keeps that result
// only when it provably equals the fp64 one:
//   |key32 - key64| <= DELTA = 5e-7 + 1.25e-7 * max|key32| for every expert
// (the fast e^-l is documented within 2 + floor(1.173 |l|) ulp, a relative
// error that moves s = 1 / (1 + e^-l) by at most s (1 - s) times it, below
// 7.5e-8 for every l; 1 + e^-l rounds once, 6e-8 in s; the fast division is
// documented within 2 ulp, 2.4e-7 at s <= 1, and returns 0 for divisors above
// 2^126, where s < 2^-126; so the sigmoid is within 3.8e-7 of its value;
// adding the bias rounds once more, 2^-24 |key|; fp64 keys are exact to
// 1e-15).  A group score (sum of the
// group's top GK keys) is then within GK * (DELTA + 1.25e-7 * max|gs|) of the
// fp64 one, since a top-m sum moves by at most m times the largest change of
// its inputs.  If the fp32 gap between the last kept and the first dropped
// group exceeds twice that bound, and the gap between each of the K + 1 best
// eligible experts and the next exceeds 2 * DELTA, the fp64 selection is the
// same set in the same order; otherwise the warp path gives fp64 keys to the
// candidates that can cross the decision (and the team kernel hands the
// token to the warp path).
//
// Warp path: each lane holds VPL consecutive experts (e = lane*VPL + j), and
// the weights of the K selected experts of TB = 32 / K tokens are computed
// together, one (token, k) per lane.
#include <cfloat>
#include <cmath>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "router_grad.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // warps per block
constexpr unsigned kFull = 0xffffffffu;
constexpr float kDeltaAbs = 5e-7f;
constexpr float kDeltaRel = 1.25e-7f;

// A float-float value hi + lo (see the routing weights below).
struct FF {
  float hi, lo;
};

struct RouteArgs {
  const float* logits;
  const float* bias;
  int T, E, K;
  int G, TG, GK;
  int renorm;
  int vec4;
  int fast;  // the fp32 selection applies to this configuration
  double scale;
  FF scale_ff;      // scale as float-float
  int scale_ff_ok;  // scale is 0 or within [2^-60, 2^60] in magnitude, exact to 2^-48 as FF
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

// One logit of row t as the selection sees it (NaN as -inf).
__device__ __forceinline__ float logit_at(const RouteArgs& a, int t, int e) {
  const float x = __ldg(a.logits + static_cast<size_t>(t) * a.E + e);
  return isnan(x) ? -INFINITY : x;
}

template <int VPL>
__device__ __forceinline__ void reload_logits(const RouteArgs& a, int t, int lane, float (&v)[VPL]) {
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane * VPL + j;
    v[j] = e < a.E ? logit_at(a, t, e) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// reference-precision paths, one token at a time (all lanes take part)

// Sigmoid routing of token t entirely in fp64 (keys, group scores,
// selection and weights); writes idx and w.  wkeys: E doubles of shared
// memory owned by this warp.
template <int VPL>
__device__ void sigmoid_token_fp64(const RouteArgs& a, int t, int lane, double* wkeys) {
  float v[VPL];
  reload_logits<VPL>(a, t, lane, v);
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
__device__ void softmax_token_full(const RouteArgs& a, int t, int lane) {
  float v[VPL];
  reload_logits<VPL>(a, t, lane, v);
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

// The top two keys of a group whose keys are spread over L lanes (each
// lane's list sorted), merged over lane bits 1..L/2.
__device__ __forceinline__ void group_top2_fp32(float& t0, float& t1, int lanes) {
  for (int off = 1; off < lanes; off <<= 1) {
    const float o0 = __shfl_xor_sync(kFull, t0, off);
    const float o1 = __shfl_xor_sync(kFull, t1, off);
    const float n0 = fmaxf(t0, o0);
    const float n1 = fmaxf(fminf(t0, o0), fmaxf(t1, o1));
    t0 = n0;
    t1 = n1;
  }
}

// fp64 -> uint64 with the same order (no NaN reaches here)
__device__ __forceinline__ uint64_t order_key64(double d) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// Lane holding the largest key among the lanes where `valid` is set, the
// lowest such lane on ties; -1 if no lane is valid.  Integer reductions only.
__device__ __forceinline__ int warp_argmax_u64(bool valid, uint64_t key) {
  const uint32_t hi = valid ? static_cast<uint32_t>(key >> 32) : 0u;
  const uint32_t mhi = __reduce_max_sync(kFull, hi);
  const bool c1 = valid && hi == mhi;
  const uint32_t lo = c1 ? static_cast<uint32_t>(key) : 0u;
  const uint32_t mlo = __reduce_max_sync(kFull, lo);
  const uint32_t who = __ballot_sync(kFull, c1 && static_cast<uint32_t>(key) == mlo);
  return who ? __ffs(who) - 1 : -1;
}

// The fp64 selection key of expert e with logit l (the reference definition).
__device__ __forceinline__ double key_fp64(const RouteArgs& a, int e, float l) {
  const double s = 1.0 / (1.0 + exp(-static_cast<double>(l)));
  return s + (a.bias ? static_cast<double>(__ldg(a.bias + e)) : 0.0);
}

// The fp32 selection key (sigmoid + bias), the same expression everywhere:
// the fast exponential and the fast division (their documented error bounds
// enter DELTA above).
__device__ __forceinline__ float sigmoid_key(float l, float b) {
  const float s = __fdividef(1.0f, __fadd_rn(1.0f, __expf(-l)));
  return __fadd_rn(s, b);
}

__device__ __forceinline__ float key_fp32(const RouteArgs& a, int e, float l) {
  return sigmoid_key(l, a.bias ? __ldg(a.bias + e) : 0.0f);
}

// Gathers the lanes' candidate experts (bit j of `mask`: expert lane*VPL + j)
// into the warp's list in expert order and hands candidate i to lane i.
// Returns the count (the same in every lane), or -1 if it exceeds 32.
template <int VPL>
__device__ __forceinline__ int compact_candidates(const RouteArgs& a, int t, uint32_t mask, int lane,
                                                  int2* list, int2& mine) {
  const int c = __popc(mask);
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += o;
  }
  const int total = __shfl_sync(kFull, incl, 31);
  if (total > 32) return -1;
  int o = incl - c;
#pragma unroll
  for (int j = 0; j < VPL; ++j)
    if ((mask >> j) & 1u) {
      const int e = lane * VPL + j;
      list[o++] = make_int2(e, __float_as_int(logit_at(a, t, e)));
    }
  __syncwarp();
  mine = lane < total ? list[lane] : make_int2(0, 0);
  __syncwarp();
  return total;
}

// Selection of one token from fp32 keys.  Returns true with the k-th
// selected expert in lane base + k, or false if the token needs the full fp64
// path.  Where an fp32 decision is closer than its error bound, only the
// candidates that can cross it get fp64 keys:
//   experts: an eligible expert whose fp32 key is more than 2 * DELTA below
//     the K-th pick's has an fp64 key below those of all K picks, so the fp64
//     top-K lies among the experts within 2 * DELTA of the K-th pick or above;
//   groups: likewise a group more than 2 * DG below the TG-th group score is
//     out, and a group's fp64 score only involves its experts within 2 * DELTA
//     of its GK-th fp32 key or above.
// The candidates (at most 32) get one fp64 key each, one per lane, and the
// selection among them uses the exact fp64 order (ties to the lower index).
template <int VPL, bool SIGMOID>
__device__ __forceinline__ bool select_fp32(const RouteArgs& a, int t, int lane, float (&sk)[VPL],
                                            int base, int& my_idx, int2* list) {
  // sk holds the lane's logits on entry and becomes its sorted keys
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
        sk[j] = key_fp32(a, e, sk[j]);
        maxabs = fmaxf(maxabs, fabsf(sk[j]));
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
    float t0 = sk[0], t1 = VPL > 1 ? sk[VPL > 1 ? 1 : 0] : -INFINITY;
    group_top2_fp32(t0, t1, L);
    const float gs = a.GK >= 2 ? __fadd_rn(__fadd_rn(0.0f, t0), t1) : t0;
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
    if (a.TG < a.G && !(last - next > 2.0f * dg)) {
      // refine the group choice with fp64 group scores of the candidate groups
      const uint32_t cg = __ballot_sync(kFull, glane && my_gs >= last - 2.0f * dg);
      uint32_t mask = 0;
      if (lane * VPL < a.E && ((cg >> ((lane * VPL) / gsz)) & 1u)) {
        const float thr = (a.GK >= 2 ? t1 : t0) - 2.0f * delta;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
          if (sk[i] >= thr && lane * VPL + sj[i] < a.E) mask |= 1u << sj[i];
      }
      int2 c;
      const int n = compact_candidates<VPL>(a, t, mask, lane, list, c);
      if (n < 0) return false;
      const bool have = lane < n;
      const double kd = have ? key_fp64(a, c.x, __int_as_float(c.y)) : 0.0;
      const uint64_t ok = order_key64(kd);
      const int cgrp = c.x / gsz;
      uint64_t my_gs64 = 0;
      for (uint32_t rem = cg; rem; rem &= rem - 1) {
        const int g = __ffs(rem) - 1;
        const int w1 = warp_argmax_u64(have && cgrp == g, ok);
        double sum = __shfl_sync(kFull, kd, w1 & 31);
        if (a.GK >= 2) {
          const int w2 = warp_argmax_u64(have && cgrp == g && lane != w1, ok);
          sum = sum + __shfl_sync(kFull, kd, w2 & 31);
        }
        if (lane == g) my_gs64 = order_key64(sum);
      }
      keep = 0;
      for (int r = 0; r < a.TG; ++r) {
        const int wg = warp_argmax_u64(glane && ((cg >> lane) & 1u) && !((keep >> lane) & 1u), my_gs64);
        keep |= 1u << (wg & 31);
      }
    }
    eligible_lane = eligible_lane && ((keep >> ((lane * VPL) / gsz)) & 1u);
  }

  // K (+1 for the gap check) rounds over the lanes' heads
  int consumed = 0;
  float prev = 0.0f, vK = 0.0f;
  bool close = false;
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
    if (SIGMOID && k > 0 && !(prev - wv > 2.0f * delta)) close = true;
    prev = wv;
    if (k == a.K - 1) vK = wv;
    if (k < a.K && lane == base + k) my_idx = wl * VPL + wj;
  }
  if (!SIGMOID || !close) return true;

  // refine the expert choice: fp64 keys for the eligible experts within
  // 2 * DELTA of the K-th pick or above
  const float thr = vK - 2.0f * delta;
  uint32_t mask = 0;
  if (eligible_lane) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane * VPL + j;
      if (e < a.E && key_fp32(a, e, logit_at(a, t, e)) >= thr) mask |= 1u << j;
    }
  }
  int2 c;
  const int n = compact_candidates<VPL>(a, t, mask, lane, list, c);
  if (n < 0) return false;
  const bool have = lane < n;
  const uint64_t ok = order_key64(have ? key_fp64(a, c.x, __int_as_float(c.y)) : 0.0);
  bool taken = false;
  for (int k = 0; k < a.K; ++k) {
    const int w = warp_argmax_u64(have && !taken, ok);
    if (lane == w) taken = true;
    const int e = __shfl_sync(kFull, c.x, w & 31);
    if (lane == base + k) my_idx = e;
  }
  return true;
}

// The weights' e^x and 1/d, accurate to about 2^-41 and 2^-46 (far below the
// half ulp of the fp32 weights they end in) with fewer fp64 instructions than
// the correctly rounded library functions; fp64 issue is the scarce resource
// of this kernel.  The selection's fp64 keys keep the library exp, since
// their order must match the reference's.
//
// e^x: Cody and Waite's range reduction x = n ln2 + r, |r| <= ln2 / 2, with
// ln2 split into a head of 32 significant bits (so that n * head is exact
// for |n| < 2^21) and the rest rounded to double; then the Taylor polynomial
// of degree 10 in Horner form, whose truncation error is below
// 0.35^11 / 11! * e^0.35 = 3e-13 relative; then the factor 2^n through the
// exponent field.  Below -708 the result is 0 (e^x < 2^-1021, far below any
// fp32 weight), above 709 infinity.
constexpr double kInvLn2 = 1.4426950408889634;
constexpr double kLn2Head = 0x1.62e42ff000000p-1;
constexpr double kLn2Tail = -0x1.718432a1b0e26p-35;

__device__ __forceinline__ double exp_weight(double x) {
  if (x != x) return x;  // NaN (-inf - -inf) stays NaN, as in the reference
  if (!(x > -708.0)) return 0.0;  // also -inf
  if (x > 709.0) return INFINITY;
  const double n = rint(x * kInvLn2);
  const double r = fma(-n, kLn2Tail, fma(-n, kLn2Head, x));
  double p = 1.0 / 3628800.0;  // 1/10!
  p = fma(p, r, 1.0 / 362880.0);
  p = fma(p, r, 1.0 / 40320.0);
  p = fma(p, r, 1.0 / 5040.0);
  p = fma(p, r, 1.0 / 720.0);
  p = fma(p, r, 1.0 / 120.0);
  p = fma(p, r, 1.0 / 24.0);
  p = fma(p, r, 1.0 / 6.0);
  p = fma(p, r, 0.5);
  p = fma(p, r, 1.0);
  p = fma(p, r, 1.0);
  const long long bits = static_cast<long long>(static_cast<int>(n) + 1023) << 52;  // 2^n, n in [-1022, 1023]
  return p * __longlong_as_double(bits);
}

// 1/d: the correctly rounded fp32 reciprocal of d rounded to fp32 (relative
// error below 2^-23), then one Newton step in fp64, which squares the error
// (below 2^-46, plus the step's own rounding).  Outside the fp32 range the
// full division.
__device__ __forceinline__ double rcp_weight(double d) {
  if (!(d > 1e-30 && d < 1e30)) return 1.0 / d;
  const double r0 = static_cast<double>(__frcp_rn(static_cast<float>(d)));
  return fma(r0, fma(-d, r0, 1.0), r0);
}

// ---------------------------------------------------------------------------
// The weights in float-float arithmetic (a value is hi + lo, two fp32 with
// |lo| <= half an ulp of hi): Dekker's and Knuth's error-free sum and product
// steps with fused multiply-add, about 2^-44 relative overall, so each fp32
// weight is the fp64 reference's rounding or one ulp from it (only where the
// exact value lies within about 2^-20 ulp of a rounding midpoint).  fp32 issues
// many times faster than fp64 on this part, which is what bounds the weights.
// Tokens with a non-finite selected logit, or sigmoid logits below -700
// (where the fp64 reference's exp overflows and its weights become 0 or
// NaN), keep the fp64 path; the decision is per warp.

__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

// |a| >= |b| (or a = 0)
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  FF s = ff_two_sum(a.hi, b.hi);
  const FF t = ff_two_sum(a.lo, b.lo);
  s = ff_fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, t.lo));
}

__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return ff_fast_two_sum(p, e);
}

// a / b for b > 0 in the normal range: the rounded quotient, then the
// quotient of the exact remainder
__device__ __forceinline__ FF ff_div(FF a, FF b) {
  const float q1 = __fdiv_rn(a.hi, b.hi);
  const float p = __fmul_rn(q1, b.hi);
  const float pe = __fmaf_rn(q1, b.hi, -p);
  float r = __fsub_rn(a.hi, p);  // exact: p is within a few ulps of a.hi
  r = __fsub_rn(r, pe);
  r = __fadd_rn(r, a.lo);
  r = __fmaf_rn(-q1, b.lo, r);
  return ff_fast_two_sum(q1, __fdiv_rn(r, b.hi));
}

// 2^e for e in [-126, 127]
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// v * 2^e for e <= 0 (both parts; what falls below the fp32 range is lost,
// which only happens to terms far below the sums they enter)
__device__ __forceinline__ FF ff_scale(FF v, int e) {
  if (e < -250) return {0.0f, 0.0f};
  const int e1 = e < -125 ? -125 : e;  // both factors within pow2f's range
  const float f1 = pow2f(e1), f2 = pow2f(e - e1);
  return {__fmul_rn(__fmul_rn(v.hi, f1), f2), __fmul_rn(__fmul_rn(v.lo, f1), f2)};
}

// The fp32 weight round(v * 2^e), e <= 0, v > 0 in the normal range: v.hi is
// v rounded to fp32, so in the normal range the scaled v.hi is the rounding;
// below it one rounding of v.hi * 2^e (the first factor keeps the product
// normal and exact)
__device__ __forceinline__ float ff_to_weight(FF v, int e) {
  if (e < -160) return 0.0f;
  const int e1 = e < -100 ? -100 : e;
  return __fmul_rn(__fmul_rn(v.hi, pow2f(e1)), pow2f(e - e1));
}

// ln 2 = kLn2A + kLn2B + kLn2C: kLn2A = 355/512 has 9 significant bits, so
// n * kLn2A is exact for |n| < 2^15
constexpr float kLn2A = 0.693359375f;
constexpr float kLn2B = -0x1.bd0106p-13f;
constexpr float kLn2C = 0x1.cf79acp-40f;
constexpr float kLog2E = 0x1.715476p+0f;

// e^r for |r| <= 0.35 (float-float r): the Taylor polynomial of degree 11,
// whose truncation error is below 0.35^12 / 12! = 2^-47; the terms of
// degree 7 and up (below 2^-12 of the sum) in plain fp32, the rest with
// float-float coefficients 1/k!
__device__ __forceinline__ FF ff_exp_reduced(FF r) {
  const FF c[7] = {{1.0f, 0.0f},
                   {1.0f, 0.0f},
                   {0.5f, 0.0f},
                   {0x1.555556p-3f, -0x1.555556p-28f},
                   {0x1.555556p-5f, -0x1.555556p-30f},
                   {0x1.111112p-7f, -0x1.dddddep-32f},
                   {0x1.6c16c2p-10f, -0x1.27d27ep-35f}};
  float t = 0x1.ae6456p-26f;  // 1/11!
  t = __fmaf_rn(t, r.hi, 0x1.27e4fcp-22f);
  t = __fmaf_rn(t, r.hi, 0x1.71de3ap-19f);
  t = __fmaf_rn(t, r.hi, 0x1.a01a02p-16f);
  t = __fmaf_rn(t, r.hi, 0x1.a01a02p-13f);
  FF p = {t, 0.0f};
#pragma unroll
  for (int k = 6; k >= 0; --k) p = ff_add(ff_mul(p, r), c[k]);
  return p;
}

// e^x = m * 2^n for x <= 0, x.hi >= -760: n = round(x / ln 2) and
// m = e^(x - n ln 2) in [0.70, 1.42]; the reduced argument is exact to
// about 2^-60 (x.hi - n kLn2A is exact, n kLn2B is split exactly)
__device__ __forceinline__ FF ff_exp_nonpos(FF x, int& n) {
  const float nf = rintf(__fmul_rn(x.hi, kLog2E));
  n = static_cast<int>(nf);
  FF r = ff_two_sum(__fmaf_rn(-nf, kLn2A, x.hi), x.lo);
  const float b = __fmul_rn(-nf, kLn2B);
  r = ff_add(r, FF{b, __fmaf_rn(-nf, kLn2B, -b)});
  r = ff_add(r, FF{__fmul_rn(-nf, kLn2C), 0.0f});
  return ff_exp_reduced(r);
}

// The token's K entries sit on lanes base .. base + K - 1.  Sum over them:
// a butterfly when K is a power of two, else in k order.
__device__ __forceinline__ FF ff_token_sum(FF v, int base, int K) {
  if ((K & (K - 1)) == 0) {
    for (int off = 1; off < K; off <<= 1)
      v = ff_add(v, FF{__shfl_xor_sync(kFull, v.hi, off), __shfl_xor_sync(kFull, v.lo, off)});
    return v;
  }
  FF s{0.0f, 0.0f};
  for (int k = 0; k < K; ++k)
    s = ff_add(s, FF{__shfl_sync(kFull, v.hi, (base + k) & 31), __shfl_sync(kFull, v.lo, (base + k) & 31)});
  return s;
}

__device__ __forceinline__ int token_max(int v, int base, int K) {
  if ((K & (K - 1)) == 0) {
    for (int off = 1; off < K; off <<= 1) v = max(v, __shfl_xor_sync(kFull, v, off));
    return v;
  }
  int m = INT_MIN;
  for (int k = 0; k < K; ++k) m = max(m, __shfl_sync(kFull, v, (base + k) & 31));
  return m;
}

// The fp32 weight of this lane's entry (logit l of the token whose entries
// sit on lanes base ..), as the fp64 definition gives it; every lane of the
// warp calls it together.
template <bool SIGMOID>
__device__ __forceinline__ float weight_ff(const RouteArgs& a, float l, int base) {
  FF m;
  int n;
  if (!SIGMOID) {
    // e^(l - l_max) / sum over the selected; l_max is the first pick, so the
    // sum is at least 1 and every exponent is <= 0
    const float top = __shfl_sync(kFull, l, base & 31);
    const FF d = ff_two_sum(l, -top);  // exact
    if (d.hi < -104.0f) {
      m = FF{0.0f, 0.0f};  // its weight is below half the smallest subnormal
      n = 0;
    } else {
      m = ff_exp_nonpos(d, n);
    }
    const FF den = ff_token_sum(ff_scale(m, n), base, a.K);
    return ff_to_weight(ff_mul(ff_div(m, den), a.scale_ff), n);
  }
  // s = 1 / (1 + e^-l) = m 2^n: for l >= 0 from e^-l, for l < 0 as
  // e^l / (1 + e^l) (no overflow)
  const FF x{-fabsf(l), 0.0f};
  int ne;
  const FF e = ff_exp_nonpos(x, ne);
  const FF onep = ff_add(FF{1.0f, 0.0f}, ff_scale(e, ne));
  if (l >= 0.0f) {
    m = ff_div(FF{1.0f, 0.0f}, onep);
    n = 0;
  } else {
    m = ff_div(e, onep);
    n = ne;
  }
  if (!a.renorm) return ff_to_weight(ff_mul(m, a.scale_ff), n);
  // s_k / sum_j s_j, each term scaled by the largest 2^n of the token
  const int N = token_max(n, base, a.K);
  const FF den = ff_token_sum(ff_scale(m, n - N), base, a.K);
  return ff_to_weight(ff_mul(ff_div(m, den), a.scale_ff), n - N);
}

// Routes the tokens t0, t0 + stride, ..., count of them (at most 32 / K),
// with the whole warp: the selection one token at a time, then the weights of
// all of them in one pass, lane j * K + k holding rank k of token j.
template <int VPL, bool SIGMOID>
__device__ __forceinline__ void warp_route_tokens(const RouteArgs& a, int t0, int stride, int count,
                                                  int lane, double* wkeys, int2* list) {
  const int j_of_lane = lane / a.K, k_of_lane = lane % a.K;
  int my_idx = 0;
  float my_logit = 0.0f;
  bool my_fast = false;
  for (int j = 0; j < count; ++j) {
    const int t = t0 + j * stride;
    float v[VPL];
    const bool bad = load_logits<VPL>(a, t, lane, v);
    if (__any_sync(kFull, bad) && lane == 0) raise_flag(a.flags, MOE_DEVERR_NONFINITE);
    // a softmax selection on fp32 logits is exact even with infinities; a
    // sigmoid token with a non-finite logit goes to the fp64 path
    const bool use_fast = a.fast && !(SIGMOID && __any_sync(kFull, bad));
    int sel_idx = 0;
    const bool ok = use_fast && select_fp32<VPL, SIGMOID>(a, t, lane, v, j * a.K, sel_idx, list);
    if (ok) {
      if (j_of_lane == j) {
        my_idx = sel_idx;
        my_logit = __ldg(a.logits + static_cast<size_t>(t) * a.E + sel_idx);
        my_fast = true;
      }
    } else if (SIGMOID) {
      sigmoid_token_fp64<VPL>(a, t, lane, wkeys);
    } else {
      softmax_token_full<VPL>(a, t, lane);
    }
  }
  // weights of the tokens selected in fp32: lane = (token j, rank k);
  // float-float unless a token of the warp has a selected logit outside its
  // range (then fp64)
  const int t = t0 + j_of_lane * stride;
  const bool in_range = isfinite(my_logit) && (!SIGMOID || my_logit >= -700.0f);
  const int base = (j_of_lane * a.K) & 31;
  float wv;
  if (a.scale_ff_ok && __all_sync(kFull, !my_fast || in_range)) {
    wv = weight_ff<SIGMOID>(a, my_fast ? my_logit : 0.0f, base);
  } else {
    double val;
    if (SIGMOID) {
      val = rcp_weight(1.0 + exp_weight(-static_cast<double>(my_logit)));
    } else {
      const float top = __shfl_sync(kFull, my_logit, base);
      val = exp_weight(static_cast<double>(my_logit) - static_cast<double>(top));
    }
    // the sum over the token's K lanes: a butterfly when K is a power of
    // two (every lane then holds the same bits), else in k order
    double den = 0.0;
    if ((a.K & (a.K - 1)) == 0) {
      den = val;
      for (int off = 1; off < a.K; off <<= 1) den += __shfl_xor_sync(kFull, den, off);
    } else {
      for (int k = 0; k < a.K; ++k) den += __shfl_sync(kFull, val, (j_of_lane * a.K + k) & 31);
    }
    const double p = (SIGMOID && !a.renorm) ? val : val * rcp_weight(den);
    wv = static_cast<float>(p * a.scale);
  }
  if (my_fast && j_of_lane < count) {
    a.idx[static_cast<size_t>(t) * a.K + k_of_lane] = my_idx;
    a.w[static_cast<size_t>(t) * a.K + k_of_lane] = wv;
  }
}

template <int VPL, bool SIGMOID>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteArgs a) {
  grid_dependency_wait();
  extern __shared__ double route_smem[];
  __shared__ int2 cand_lists[kRouteWarps][32];
  double* wkeys = route_smem + (threadIdx.x >> 5) * a.E;
  int2* list = cand_lists[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int TB = 32 / a.K;  // tokens per weight pass
  // persistent grid: warp w takes tokens w, w + W, w + 2W, ... (W warps in
  // all), TB at a time, so every warp gets the same number of tokens to
  // within one
  const int W = gridDim.x * kRouteWarps;
  const int wid = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  for (int i0 = 0; wid + i0 * W < a.T; i0 += TB) {
    const int t0 = wid + i0 * W;
    const int count = min(TB, (a.T - t0 + W - 1) / W);
    warp_route_tokens<VPL, SIGMOID>(a, t0, W, count, lane, wkeys, list);
  }
}

// ---------------------------------------------------------------------------
// Eight threads per token, where E is 64, 128 or 256, K <= 8, the rows are
// 16-byte aligned and, for group-limited sigmoid routing, a group is one,
// two, four or eight threads' experts: thread p of a token's team holds
// experts [p E/8, (p + 1) E/8) in registers, keeps its own sorted list of
// candidate words, and the team merges the lists in three butterfly rounds,
// so a token takes a few hundred instructions instead of the warp path's
// K + 1 warp-wide selection rounds.  Four tokens per warp.
//
// Each candidate is one 32-bit word, q << 8 | (255 - e), with q a 23-bit
// quantisation of its key that never ranks a smaller key above a larger one:
// the larger word has the larger q, or the same q and the lower expert, and
// no two words are equal.  A list is the 8 largest words, sorted, plus the
// largest word below them: a thread sorts its words 8 at a time (Batcher's
// odd-even merge network) and folds each sorted 8 into its list, and the
// team folds its threads' lists together, by a bitonic step: the larger of
// L[i] and B[7 - i] for each i is the top 8 as a bitonic sequence, which
// three half-cleaner stages sort, and the largest of the smaller ones (and
// of the two lists' ninth words) is the ninth.  Where the listed q strictly
// decrease, every listed key is strictly above the next and above every
// unlisted key, so the first K are the K largest keys, in order, and no two
// are equal.
//   softmax: the key is the logit and q its position in a window of width 32
//     around the largest of the row's first 8 logits, in steps of 2^-18;
//     logits outside the window clamp to its ends.
//   sigmoid: the key is the fp32 sigmoid + bias (within DELTA of the fp64
//     key), q its position in [min bias, 1 + max bias], rounded, in steps of
//     1/qs, so a key lies within half a step of its q.  Two listed keys whose
//     q differ by more than 1 + 2 DELTA qs are more than 2 DELTA apart, and
//     so are the K-th and any unlisted key when the K-th and (K+1)-th differ
//     that much; then the fp64 keys rank the same.  Group scores (the sum of
//     a group's top GK fp32 keys) are ranked exactly, ties to the lower
//     group, and the TG kept groups must be more than 2 DG above the next, as
//     in the warp path; only the kept groups' threads list their experts.
// A token that fails a test, has a non-finite logit or bias, or a selected
// sigmoid logit below -700, is routed again by its warp on the
// warp-per-token path above.  The weights are weight_ff's, lane p of the team
// holding rank p.

constexpr int kTeam = 8;       // threads per token
constexpr int kTeamWarps = 4;  // warps per block

// a >= b afterwards
__device__ __forceinline__ void cmp_desc(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b);
  b = min(a, b);
  a = hi;
}

// Batcher's odd-even merge sort of 8 words, descending (19 comparators).
__device__ __forceinline__ void sort8_desc(uint32_t (&v)[8]) {
  cmp_desc(v[0], v[1]); cmp_desc(v[2], v[3]); cmp_desc(v[4], v[5]); cmp_desc(v[6], v[7]);
  cmp_desc(v[0], v[2]); cmp_desc(v[1], v[3]); cmp_desc(v[4], v[6]); cmp_desc(v[5], v[7]);
  cmp_desc(v[1], v[2]); cmp_desc(v[5], v[6]);
  cmp_desc(v[0], v[4]); cmp_desc(v[1], v[5]); cmp_desc(v[2], v[6]); cmp_desc(v[3], v[7]);
  cmp_desc(v[2], v[4]); cmp_desc(v[3], v[5]);
  cmp_desc(v[1], v[2]); cmp_desc(v[3], v[4]); cmp_desc(v[5], v[6]);
}

// (L, l9) becomes the 8 largest words of both lists, sorted, and the ninth.
__device__ __forceinline__ void merge8(uint32_t (&L)[8], uint32_t& l9, const uint32_t (&B)[8],
                                       uint32_t b9) {
  uint32_t d = max(l9, b9);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t x = L[i], y = B[7 - i];
    L[i] = max(x, y);
    d = max(d, min(x, y));
  }
  l9 = d;
#pragma unroll
  for (int i = 0; i < 4; ++i) cmp_desc(L[i], L[i + 4]);
  cmp_desc(L[0], L[2]); cmp_desc(L[1], L[3]); cmp_desc(L[4], L[6]); cmp_desc(L[5], L[7]);
  cmp_desc(L[0], L[1]); cmp_desc(L[2], L[3]); cmp_desc(L[4], L[5]); cmp_desc(L[6], L[7]);
}

// Folds 8 words (unsorted) into the list (L, l9); `first`: the list is empty.
__device__ __forceinline__ void fold8(uint32_t (&L)[8], uint32_t& l9, uint32_t (&w)[8], bool first) {
  sort8_desc(w);
  if (first) {
#pragma unroll
    for (int i = 0; i < 8; ++i) L[i] = w[i];
    l9 = 0u;
  } else {
    merge8(L, l9, w, 0u);
  }
}

// The word of expert e whose scaled key is v = key * qs + qo: an fp32 in
// [2^23, 2^24) is 2^23 plus an integer, which is its mantissa field; v is
// clamped to that range (as bit patterns, which order like the values, with
// negative ones below) and the mantissa shifted up by 8 bits.
__device__ __forceinline__ uint32_t pack_word(float v, int e) {
  const int bits = min(max(__float_as_int(v), 0x4B000000), 0x4B7FFFFF);
  return static_cast<uint32_t>(bits) * 256u + static_cast<uint32_t>(255 - e);
}

__device__ __forceinline__ int word_expert(uint32_t w) { return 255 - static_cast<int>(w & 255u); }

template <int EP, bool SIGMOID>
__global__ void __launch_bounds__(kTeamWarps * 32) route_team_kernel(RouteArgs a) {
  grid_dependency_wait();
  extern __shared__ double route_smem[];  // the fallback's fp64 keys: E per warp (sigmoid)
  __shared__ int2 cand_lists[kTeamWarps][32];
  __shared__ __align__(16) float bias_s[256];
  __shared__ float brange[2][kTeamWarps];
  __shared__ int bias_bad;
  constexpr int VPL = EP / 4;  // the warp path's experts per lane for this E
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int p = lane & (kTeam - 1), base = lane & ~(kTeam - 1);
  double* wkeys = route_smem + warp * a.E;
  int2* list = cand_lists[warp];

  // sigmoid: the bias (shared), and the scaling of keys to words from its range
  float qs = 0.0f, qo = 0.0f;
  bool bias_ok = true;
  if (SIGMOID) {
    if (threadIdx.x == 0) bias_bad = 0;
    __syncthreads();
    float bmin = INFINITY, bmax = -INFINITY;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
      const float b = a.bias ? __ldg(a.bias + e) : 0.0f;
      bias_s[e] = b;
      if (!isfinite(b)) bias_bad = 1;
      bmin = fminf(bmin, b);
      bmax = fmaxf(bmax, b);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      bmin = fminf(bmin, __shfl_xor_sync(kFull, bmin, off));
      bmax = fmaxf(bmax, __shfl_xor_sync(kFull, bmax, off));
    }
    if (lane == 0) {
      brange[0][warp] = bmin;
      brange[1][warp] = bmax;
    }
    __syncthreads();
    bmin = brange[0][0];
    bmax = brange[1][0];
    for (int w = 1; w < kTeamWarps; ++w) {
      bmin = fminf(bmin, brange[0][w]);
      bmax = fmaxf(bmax, brange[1][w]);
    }
    bias_ok = bias_bad == 0;
    qs = 0x1p23f / __fsub_rn(__fadd_rn(1.0f, bmax), bmin);
    qo = __fmaf_rn(-bmin, qs, 0x1p23f);
  }
  const int gsz = a.E / a.G;
  const int m = SIGMOID && a.G > 1 ? gsz / EP : 1;  // threads per group
  const int n_elig = SIGMOID && a.G > 1 ? a.TG * gsz : a.E;
  const int n_list = a.K < n_elig ? a.K + 1 : a.K;

  const int stride = gridDim.x * kTeamWarps * (32 / kTeam);
  for (int t0 = (blockIdx.x * kTeamWarps + warp) * (32 / kTeam); t0 < a.T; t0 += stride) {
    const int t = t0 + lane / kTeam;
    const bool active = t < a.T;
    const float* row = a.logits + static_cast<size_t>(active ? t : t0) * a.E;
    float kx[EP];
#pragma unroll
    for (int c = 0; c < EP; c += 4) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + p * EP + c));
      kx[c] = f.x;
      kx[c + 1] = f.y;
      kx[c + 2] = f.z;
      kx[c + 3] = f.w;
    }
    float fin = 0.0f;  // NaN once a logit of the token is not finite
#pragma unroll
    for (int c = 0; c < EP; ++c) fin = __fmaf_rn(kx[c], 0.0f, fin);
    uint32_t L[8], l9;
    bool ok = active && bias_ok;
    float gap = 0.0f;  // q difference a listed pair must exceed (sigmoid)
    if (!SIGMOID) {
      float m0 = kx[0];
#pragma unroll
      for (int c = 1; c < 8; ++c) m0 = fmaxf(m0, kx[c]);
      m0 = __shfl_sync(kFull, m0, base);
      const float so = __fmaf_rn(-__fsub_rn(m0, 16.0f), 0x1p18f, 0x1p23f);
#pragma unroll
      for (int b = 0; b < EP; b += 8) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = pack_word(__fmaf_rn(kx[b + j], 0x1p18f, so), p * EP + b + j);
        fold8(L, l9, w, b == 0);
      }
    } else {
      float maxabs = 0.0f, t0v = -INFINITY, t1v = -INFINITY;
#pragma unroll
      for (int c = 0; c < EP; c += 4) {
        const float4 b = *reinterpret_cast<const float4*>(bias_s + p * EP + c);
        kx[c] = sigmoid_key(kx[c], b.x);
        kx[c + 1] = sigmoid_key(kx[c + 1], b.y);
        kx[c + 2] = sigmoid_key(kx[c + 2], b.z);
        kx[c + 3] = sigmoid_key(kx[c + 3], b.w);
      }
#pragma unroll
      for (int c = 0; c < EP; ++c) {
        maxabs = fmaxf(maxabs, fabsf(kx[c]));
        const float n0 = fmaxf(t0v, kx[c]);
        t1v = fmaxf(t1v, fminf(t0v, kx[c]));
        t0v = n0;
      }
#pragma unroll
      for (int off = 1; off < kTeam; off <<= 1)
        maxabs = fmaxf(maxabs, __shfl_xor_sync(kFull, maxabs, off));
      const float delta = kDeltaAbs + kDeltaRel * maxabs;
      ok = ok && delta < 1e-3f;  // huge or non-finite keys fail here
      gap = __fmaf_rn(2.0f * delta, qs, 1.0f);
      bool kept = true;
      if (a.G > 1) {
        // the group's top two over its m threads, then its score
        group_top2_fp32(t0v, t1v, m);
        const float gs = a.GK >= 2 ? __fadd_rn(__fadd_rn(0.0f, t0v), t1v) : t0v;
        const int g = p / m;
        int rank = 0;  // groups ranked before this one (score desc, group asc)
        float gmax = 0.0f;
        for (int j = 0; j < a.G; ++j) {
          const float sj = __shfl_sync(kFull, gs, base + j * m);
          gmax = fmaxf(gmax, fabsf(sj));
          if (sj > gs || (sj == gs && j < g)) ++rank;
        }
        kept = rank < a.TG;
        if (a.TG < a.G) {
          // the lowest kept score must clear the highest dropped one
          float last = kept ? gs : INFINITY, next = kept ? -INFINITY : gs;
#pragma unroll
          for (int off = 1; off < kTeam; off <<= 1) {
            last = fminf(last, __shfl_xor_sync(kFull, last, off));
            next = fmaxf(next, __shfl_xor_sync(kFull, next, off));
          }
          const float dg = a.GK * (delta + kDeltaRel * gmax);
          ok = ok && last - next > 2.0f * dg;
        }
      }
#pragma unroll
      for (int b = 0; b < EP; b += 8) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = pack_word(__fmaf_rn(kx[b + j], qs, qo), p * EP + b + j);
        fold8(L, l9, w, b == 0);
      }
      if (!kept) {  // a dropped group's experts are not candidates
#pragma unroll
        for (int i = 0; i < 8; ++i) L[i] = 0u;
        l9 = 0u;
      }
    }
    // the team's lists merged: every thread of the team ends with the same list
#pragma unroll
    for (int off = 1; off < kTeam; off <<= 1) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(kFull, L[i], off);
      merge8(L, l9, o, __shfl_xor_sync(kFull, l9, off));
      fin = __fadd_rn(fin, __shfl_xor_sync(kFull, fin, off));
    }
    // the listed q strictly decrease, for sigmoid by more than the gap
#pragma unroll
    for (int i = 1; i <= 8; ++i) {
      if (i >= n_list) break;
      const uint32_t hi = L[i - 1], lo = i < 8 ? L[i] : l9;
      const float d = static_cast<float>(static_cast<int>(hi >> 8) - static_cast<int>(lo >> 8));
      if (SIGMOID ? !(d > gap) : !(d > 0.0f)) ok = false;
    }
    ok = ok && fin == 0.0f;
    // rank p of the token: its expert, logit and weight
    int my_e = 0;
#pragma unroll
    for (int i = 0; i < kTeam; ++i)
      if (i == p) my_e = word_expert(L[i]);
    const bool mine = p < a.K;
    const float l = mine ? __ldg(row + my_e) : 0.0f;
    if (SIGMOID && mine && !(l >= -700.0f)) ok = false;  // the fp64 path's range
    // every test so far gave the whole team one answer, except that range test: share it
    ok = (__ballot_sync(kFull, !ok) & (0xffu << base)) == 0;
    const float wv = weight_ff<SIGMOID>(a, ok ? l : 0.0f, base);
    if (ok && mine) {
      a.idx[static_cast<size_t>(t) * a.K + p] = my_e;
      a.w[static_cast<size_t>(t) * a.K + p] = wv;
    }
    // the tokens that failed a test, one at a time by the whole warp
    for (uint32_t fb = __ballot_sync(kFull, active && !ok && p == 0); fb; fb &= fb - 1)
      warp_route_tokens<VPL, SIGMOID>(a, t0 + (__ffs(fb) - 1) / kTeam, 0, 1, lane, wkeys, list);
  }
}

// Whether the eight-threads-per-token kernel applies (else the warp kernel).
bool team_path(const RouteArgs& a, bool sigmoid) {
  if ((a.E != 64 && a.E != 128 && a.E != 256) || a.K > kTeam || !a.vec4 || !a.scale_ff_ok) return false;
  if (!sigmoid) return a.renorm != 0;
  if (a.G == 1) return true;
  const int ep = a.E / kTeam, gsz = a.E / a.G;
  const int m = gsz / ep;
  return a.GK <= 2 && gsz % ep == 0 && (m & (m - 1)) == 0;
}

template <int EP, bool SIGMOID>
void launch_team(const RouteArgs& a, int num_sms, cudaStream_t s) {
  auto k = route_team_kernel<EP, SIGMOID>;
  const size_t smem = SIGMOID ? static_cast<size_t>(kTeamWarps) * a.E * sizeof(double) : 0;
  const int per_block = kTeamWarps * (32 / kTeam);
  const long long blocks_needed = (static_cast<long long>(a.T) + per_block - 1) / per_block;
  long long grid = static_cast<long long>(resident_blocks(reinterpret_cast<const void*>(k),
                                                          kTeamWarps * 32, smem)) * num_sms;
  if (blocks_needed < grid) grid = blocks_needed;
  (void)launch_chained(k, dim3(static_cast<int>(grid < 1 ? 1 : grid)), dim3(kTeamWarps * 32), smem, s, false, a);
}

// One wave of resident blocks (or fewer if there are fewer tokens): a second,
// partial wave would leave most SMs idle for a whole block's duration.
template <int VPL, bool SIGMOID>
void launch_one(const RouteArgs& a, int num_sms, size_t smem, cudaStream_t s) {
  auto k = route_kernel<VPL, SIGMOID>;
  const int TB = 32 / a.K;
  const long long warps_needed = (static_cast<long long>(a.T) + TB - 1) / TB;
  const long long blocks_needed = (warps_needed + kRouteWarps - 1) / kRouteWarps;
  long long grid = static_cast<long long>(resident_blocks(reinterpret_cast<const void*>(k),
                                                          kRouteWarps * 32, smem)) * num_sms;
  if (blocks_needed < grid) grid = blocks_needed;
  (void)launch_chained(k, dim3(static_cast<int>(grid < 1 ? 1 : grid)), dim3(kRouteWarps * 32), smem, s, false, a);
}

// ---------------------------------------------------------------------------
// Router backward to the logits: the per-entry derivative is
// router_grad_entry (router_grad.cuh), rounded once to fp32; every other entry
// of the row is 0.  Lane j*K + k handles entry k of token j, TB = 32/K tokens
// per warp pass.  Softmax without renormalisation moves every logit of the
// row, dL/dl_e = c p_e (gw_e - sum_k p_k gw_k) with p the full softmax and
// gw_e = 0 for unselected e; it has its own kernel below.

struct RouteBwdArgs {
  const float* logits;
  const int32_t* idx;
  const float* gw;
  float* glogits;
  int T, E, K;
  int sigmoid, renorm;
  double scale;
};

__global__ void __launch_bounds__(kRouteWarps * 32) route_bwd_kernel(RouteBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int TB = 32 / a.K;
  const int W = gridDim.x * kRouteWarps;
  const int wid = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  const int j = lane / a.K, k = lane % a.K;
  const bool vec4 = (a.E & 3) == 0 && ((reinterpret_cast<uintptr_t>(a.glogits) & 15) == 0);
  for (int i0 = 0; wid + i0 * W < a.T; i0 += TB) {
    // zero the TB rows
    for (int jj = 0; jj < TB; ++jj) {
      const int t = wid + (i0 + jj) * W;
      if (t >= a.T) break;
      float* row = a.glogits + static_cast<size_t>(t) * a.E;
      if (vec4) {
        for (int e = lane * 4; e < a.E; e += 128)
          *reinterpret_cast<float4*>(row + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int e = lane; e < a.E; e += 32) row[e] = 0.f;
      }
    }
    const int t = wid + (i0 + j) * W;
    const bool valid = j < TB && t < a.T;
    int e = 0;
    double l = 0.0, g = 0.0;
    if (valid) {
      e = __ldg(a.idx + static_cast<size_t>(t) * a.K + k);
      if (e < 0 || e >= a.E) e = 0;  // invalid indices: routed tokens come from route_topk
      l = static_cast<double>(__ldg(a.logits + static_cast<size_t>(t) * a.E + e));
      g = static_cast<double>(__ldg(a.gw + static_cast<size_t>(t) * a.K + k));
    }
    const int b = (j * a.K) & 31;  // lane of entry 0 of this token
    const double out = router_grad_entry(l, g, b, a.K, a.sigmoid, a.renorm, a.scale);
    __syncwarp();  // the zero fill above is ordered before these writes
    if (valid) a.glogits[static_cast<size_t>(t) * a.E + e] = static_cast<float>(out);
    __syncwarp();
  }
}

// softmax without renormalisation: every logit of the row moves (one token per
// warp, each lane its VPL experts)
template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_bwd_full_softmax_kernel(RouteBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * kRouteWarps;
  for (int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5); t < a.T; t += W) {
    const float* row = a.logits + static_cast<size_t>(t) * a.E;
    double m = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < VPL; ++jj) {
      const int e = lane * VPL + jj;
      if (e < a.E) m = fmax(m, static_cast<double>(__ldg(row + e)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmax(m, __shfl_xor_sync(kFull, m, off));
    double part = 0.0;
#pragma unroll
    for (int jj = 0; jj < VPL; ++jj) {
      const int e = lane * VPL + jj;
      if (e < a.E) part += exp(static_cast<double>(__ldg(row + e)) - m);
    }
    double den = 0.0;
    for (int ll = 0; ll < 32; ++ll) den += __shfl_sync(kFull, part, ll);
    double dot = 0.0;
    for (int kk = 0; kk < a.K; ++kk) {
      int e = __ldg(a.idx + static_cast<size_t>(t) * a.K + kk);
      if (e < 0 || e >= a.E) e = 0;
      dot += exp(static_cast<double>(__ldg(row + e)) - m) / den *
             static_cast<double>(__ldg(a.gw + static_cast<size_t>(t) * a.K + kk));
    }
#pragma unroll
    for (int jj = 0; jj < VPL; ++jj) {
      const int e = lane * VPL + jj;
      if (e >= a.E) continue;
      double ge = 0.0;
      for (int kk = 0; kk < a.K; ++kk)
        if (__ldg(a.idx + static_cast<size_t>(t) * a.K + kk) == e)
          ge = static_cast<double>(__ldg(a.gw + static_cast<size_t>(t) * a.K + kk));
      const double p = exp(static_cast<double>(__ldg(row + e)) - m) / den;
      a.glogits[static_cast<size_t>(t) * a.E + e] = static_cast<float>(a.scale * p * (ge - dot));
    }
  }
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
  {
    const double sc = c.route_scale;
    const float sh = static_cast<float>(sc);
    a.scale_ff = FF{sh, static_cast<float>(sc - static_cast<double>(sh))};
    a.scale_ff_ok = sc == 0.0 || (std::fabs(sc) >= 0x1p-60 && std::fabs(sc) <= 0x1p60);
  }
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
  if (team_path(a, sigmoid)) {
    switch (a.E) {
      case 64: sigmoid ? launch_team<8, true>(a, h->num_sms, s) : launch_team<8, false>(a, h->num_sms, s); break;
      case 128: sigmoid ? launch_team<16, true>(a, h->num_sms, s) : launch_team<16, false>(a, h->num_sms, s); break;
      default: sigmoid ? launch_team<32, true>(a, h->num_sms, s) : launch_team<32, false>(a, h->num_sms, s); break;
    }
    return cudaGetLastError();
  }
  const size_t smem = sigmoid && a.G > 1 ? static_cast<size_t>(kRouteWarps) * a.E * sizeof(double) : 0;
  switch (vpl) {
    case 1: sigmoid ? launch_one<1, true>(a, h->num_sms, smem, s) : launch_one<1, false>(a, h->num_sms, smem, s); break;
    case 2: sigmoid ? launch_one<2, true>(a, h->num_sms, smem, s) : launch_one<2, false>(a, h->num_sms, smem, s); break;
    case 4: sigmoid ? launch_one<4, true>(a, h->num_sms, smem, s) : launch_one<4, false>(a, h->num_sms, smem, s); break;
    case 8: sigmoid ? launch_one<8, true>(a, h->num_sms, smem, s) : launch_one<8, false>(a, h->num_sms, smem, s); break;
    default: sigmoid ? launch_one<16, true>(a, h->num_sms, smem, s) : launch_one<16, false>(a, h->num_sms, smem, s); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_route_bwd(const moe_handle* h, const float* logits, const int32_t* idx,
                             const float* gw, int T, float* glogits, cudaStream_t s) {
  const moe_config& c = h->cfg;
  RouteBwdArgs a;
  a.logits = logits;
  a.idx = idx;
  a.gw = gw;
  a.glogits = glogits;
  a.T = T;
  a.E = c.num_experts;
  a.K = c.top_k;
  a.sigmoid = c.score_fn == MOE_SCORE_SIGMOID;
  a.renorm = c.renorm;
  a.scale = c.route_scale;
  if (T == 0) return cudaSuccess;
  const int threads = kRouteWarps * 32;
  if (!a.sigmoid && !a.renorm) {
    const int vpl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : a.E <= 256 ? 8 : 16;
    const long long blocks = (static_cast<long long>(T) + kRouteWarps - 1) / kRouteWarps;
    const int grid = static_cast<int>(blocks < h->num_sms * 8 ? blocks : h->num_sms * 8);
    switch (vpl) {
      case 1: route_bwd_full_softmax_kernel<1><<<grid, threads, 0, s>>>(a); break;
      case 2: route_bwd_full_softmax_kernel<2><<<grid, threads, 0, s>>>(a); break;
      case 4: route_bwd_full_softmax_kernel<4><<<grid, threads, 0, s>>>(a); break;
      case 8: route_bwd_full_softmax_kernel<8><<<grid, threads, 0, s>>>(a); break;
      default: route_bwd_full_softmax_kernel<16><<<grid, threads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
  }
  const int TB = 32 / a.K;
  const long long warps_needed = (static_cast<long long>(T) + TB - 1) / TB;
  const long long blocks_needed = (warps_needed + kRouteWarps - 1) / kRouteWarps;
  long long grid = static_cast<long long>(resident_blocks(
                       reinterpret_cast<const void*>(route_bwd_kernel), threads, 0)) * h->num_sms;
  if (blocks_needed < grid) grid = blocks_needed;
  route_bwd_kernel<<<static_cast<int>(grid < 1 ? 1 : grid), threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
