// Top-K routing, one warp per token (sm_103a).
//
// Softmax routing selects the K largest logits (softmax is strictly
// increasing, so the set and order equal those of the probabilities) and
// weights them by softmax; group-limited sigmoid routing selects on
// key = sigmoid(logit) + score-correction bias in fp64 and weights by the
// unbiased sigmoid (DeepSpeed "Avoid collective token preparation for AutoEP
// DeepEP", "Testing Done": exact routes, score-correction bias).  Selection
// order is descending key; equal keys go to the lower expert index.  Weights
// are computed in fp64 and rounded once to fp32.
//
// Each lane holds VPL consecutive experts (e = lane*VPL + j).  A selection
// round takes the best entry strictly after the previous pick in the total
// order (key descending, index ascending), reduced across the warp with
// shuffles, so no per-entry "taken" state is needed.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // tokens in flight per block
constexpr unsigned kFull = 0xffffffffu;

struct RouteArgs {
  const float* logits;
  const float* bias;
  int T, E, K;
  int G, TG, GK;
  int renorm;
  int vec4;
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

// Loads the lane's VPL logits of row t; entries past E read as -inf.
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

template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_softmax_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * kRouteWarps;
  for (int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5); t < a.T; t += nwarps) {
    float v[VPL];
    const bool bad = load_logits<VPL>(a, t, lane, v);
    if (__any_sync(kFull, bad) && lane == 0) raise_flag(a.flags, MOE_DEVERR_NONFINITE);

    float pv = INFINITY, myv = 0.f;
    int pi = -1, myi = 0;
    for (int k = 0; k < a.K; ++k) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane * VPL + j;
        if (comes_after(v[j], e, pv, pi) && ranks_before(v[j], e, bv, bi)) {
          bv = v[j];
          bi = e;
        }
      }
      warp_best(bv, bi);
      pv = bv;
      pi = bi;
      if (lane == k) {
        myv = bv;
        myi = bi;
      }
    }

    const double lmax = static_cast<double>(__shfl_sync(kFull, myv, 0));
    const double ex = lane < a.K ? exp(static_cast<double>(myv) - lmax) : 0.0;
    double den = 0.0;
    if (a.renorm) {
      for (int k = 0; k < a.K; ++k) den += __shfl_sync(kFull, ex, k);
    } else {
      double part = 0.0;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (lane * VPL + j < a.E) part += exp(static_cast<double>(v[j]) - lmax);
      for (int l = 0; l < 32; ++l) den += __shfl_sync(kFull, part, l);
    }
    if (lane < a.K) {
      a.idx[static_cast<size_t>(t) * a.K + lane] = myi;
      a.w[static_cast<size_t>(t) * a.K + lane] = static_cast<float>((ex / den) * a.scale);
    }
  }
}

template <int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_sigmoid_kernel(RouteArgs a) {
  extern __shared__ double route_smem[];
  double* wkeys = route_smem + (threadIdx.x >> 5) * a.E;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * kRouteWarps;
  const int gsz = a.E / a.G;
  for (int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5); t < a.T; t += nwarps) {
    float v[VPL];
    const bool bad = load_logits<VPL>(a, t, lane, v);
    if (__any_sync(kFull, bad) && lane == 0) raise_flag(a.flags, MOE_DEVERR_NONFINITE);

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

    uint32_t keep = 0xffffffffu;  // eligible groups
    if (a.G > 1) {
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (lane * VPL + j < a.E) wkeys[lane * VPL + j] = key[j];
      __syncwarp();
      double gscore = -INFINITY;
      if (lane < a.G) {
        // sum of the group's top-GK keys, added in descending order
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

  const int blocks_needed = (T + kRouteWarps - 1) / kRouteWarps;
  const int cap = h->num_sms * 16;
  const int grid = blocks_needed < cap ? blocks_needed : cap;
  const int vpl = a.E <= 32 ? 1 : a.E <= 64 ? 2 : a.E <= 128 ? 4 : a.E <= 256 ? 8 : 16;
  const dim3 block(kRouteWarps * 32);
  if (c.score_fn == MOE_SCORE_SOFTMAX) {
    switch (vpl) {
      case 1: route_softmax_kernel<1><<<grid, block, 0, s>>>(a); break;
      case 2: route_softmax_kernel<2><<<grid, block, 0, s>>>(a); break;
      case 4: route_softmax_kernel<4><<<grid, block, 0, s>>>(a); break;
      case 8: route_softmax_kernel<8><<<grid, block, 0, s>>>(a); break;
      default: route_softmax_kernel<16><<<grid, block, 0, s>>>(a); break;
    }
  } else {
    const size_t smem = a.G > 1 ? static_cast<size_t>(kRouteWarps) * a.E * sizeof(double) : 0;
    switch (vpl) {
      case 1: route_sigmoid_kernel<1><<<grid, block, smem, s>>>(a); break;
      case 2: route_sigmoid_kernel<2><<<grid, block, smem, s>>>(a); break;
      case 4: route_sigmoid_kernel<4><<<grid, block, smem, s>>>(a); break;
      case 8: route_sigmoid_kernel<8><<<grid, block, smem, s>>>(a); break;
      default: route_sigmoid_kernel<16><<<grid, block, smem, s>>>(a); break;
    }
  }
  return cudaGetLastError();
}

}  // namespace moe
