// Router backward to the logits for one (token, k) entry per lane (sm_103a).
//
// DeepSpeed "Avoid collective token preparation for AutoEP DeepEP", "Testing
// Done": routing-score and router-parameter gradients.  With the selection
// fixed, the weights are
//   softmax, renorm:     w_k = c q_k,   q_k = exp(l_k) / sum_{j in sel} exp(l_j)
//   sigmoid, renorm:     w_k = c s_k / S,  S = sum_{j in sel} s_j
//   sigmoid, no renorm:  w_k = c s_k
// (the correction bias selects only and gets no gradient), so
//   softmax renorm:     dL/dl_j = c q_j (gw_j - sum_k q_k gw_k)
//   sigmoid renorm:     dL/dl_j = s_j (1 - s_j) (c / S) (gw_j - sum_k gw_k s_k / S)
//   sigmoid no renorm:  dL/dl_j = c gw_j s_j (1 - s_j)
// in fp64 with sums in k order.  Softmax without renormalisation moves every
// logit of the row and is not handled here.
//
// The work splits into what depends on the logits only (router_grad_prep:
// the exponentials and the selected-set sums) and the short rest that needs
// gw (router_grad_finish), so a caller can prepare a token before its gw is
// known.  The K entries of a token sit on lanes base .. base + K - 1 of the
// warp (base + K <= 32); every lane of the warp calls both together
// (full-warp shuffles), lanes outside a token with any finite l and g.
#pragma once

#include <cuda_runtime.h>

namespace moe {

struct RouterGradPrep {
  double p;  // softmax: q; sigmoid: s
  double S;  // sigmoid with renormalisation: the sum of the selected s
};

__device__ __forceinline__ RouterGradPrep router_grad_prep(double l, int base, int K,
                                                           bool sigmoid, bool renorm) {
  constexpr unsigned full = 0xffffffffu;
  RouterGradPrep r{0.0, 1.0};
  if (!sigmoid) {
    const double lmax = __shfl_sync(full, l, base);
    const double ex = exp(l - lmax);
    double den = 0.0;
    for (int kk = 0; kk < K; ++kk) den += __shfl_sync(full, ex, (base + kk) & 31);
    r.p = ex / den;
    return r;
  }
  r.p = 1.0 / (1.0 + exp(-l));
  if (renorm) {
    double S = 0.0;
    for (int kk = 0; kk < K; ++kk) S += __shfl_sync(full, r.p, (base + kk) & 31);
    r.S = S;
  }
  return r;
}

__device__ __forceinline__ double router_grad_finish(const RouterGradPrep& r, double g, int base,
                                                     int K, bool sigmoid, bool renorm,
                                                     double scale) {
  constexpr unsigned full = 0xffffffffu;
  if (!sigmoid) {
    const double q = r.p;
    const double qg = q * g;
    double dot = 0.0;
    for (int kk = 0; kk < K; ++kk) dot += __shfl_sync(full, qg, (base + kk) & 31);
    return scale * q * (g - dot);
  }
  const double sg = r.p;
  if (!renorm) return scale * g * sg * (1.0 - sg);
  const double S = r.S;
  const double t = g * sg / S;
  double dot = 0.0;
  for (int kk = 0; kk < K; ++kk) dot += __shfl_sync(full, t, (base + kk) & 31);
  return sg * (1.0 - sg) * (scale / S) * (g - dot);
}

__device__ __forceinline__ double router_grad_entry(double l, double g, int base, int K,
                                                    bool sigmoid, bool renorm, double scale) {
  return router_grad_finish(router_grad_prep(l, base, K, sigmoid, renorm), g, base, K, sigmoid,
                            renorm, scale);
}

}  // namespace moe
