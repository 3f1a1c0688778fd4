// CPU oracle for the MoE token dispatch / combine path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
// calls this file.  It is loaded by the tests, by the smoke check and by the
// benchmark's CPU-baseline leg, and by nothing else.
//
// Plain, slow, single-threaded C++17.  Every function follows the definition
// of one step of the method in the order the sources state it; there is no
// blocking, fusion or reordering.  It shares no code, header or constant with
// the CUDA library.
//
// Sources (web pages on MoE token dispatchers):
//   [AutoEP-DeepEP]   DeepSpeed PR "Add an opt-in DeepEP transport for the
//                     AutoEP expert all-to-all", sections "Why" and the squashed
//                     review-fix commit text.
//   [AutoEP-prep]     DeepSpeed PR "Avoid collective token preparation for
//                     AutoEP DeepEP", "Summary" and "Testing Done".
//   [Titan-absorb]    torchtitan issue "[MoE] Apply router scores before W2
//                     projection", "Motivation", "Implementation", "Tests".
//   [NeMo-DeepEPv2]   NeMo Automodel PR "DeepEP v2 dispatcher ...",
//                     "Performance" (paired handle) and "Validation".
//
// Readings where the pages are silent (each one is also listed in the design
// notes):
//   * routing math: softmax top-k renormalised; or sigmoid scores with a
//     score-correction bias that enters only the selection key, group-limited
//     (group score = sum of the top `group_score_topk` keys of the group);
//   * ties in any selection go to the lower index;
//   * softmax selection is taken on the raw logits (softmax is strictly
//     increasing, so the top-k set and order are the same), the sigmoid
//     selection on fp64 keys; weights are computed in fp64 and rounded once to
//     fp32;
//   * receive layout: expert-major, stable by token (then k);
//   * send layout: rank-major, each token once per destination rank, stable by
//     token;
//   * combine accumulates in fp32 in k order (fused multiply-add for the
//     weighted sum) and rounds once to the row dtype;
//   * an index entry outside [0, E) or repeating an expert already listed
//     earlier for the same token is dropped: it gets pos = -1, is not counted
//     and contributes nothing.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

enum { DT_BF16 = 0, DT_F32 = 1 };

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round-to-nearest-even of an fp32 value to bfloat16 (8-bit significand):
// keep the upper 16 bits, rounding on the lower 16, ties to an even result.
uint16_t float_to_bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u)  // NaN: keep it a quiet NaN
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
  return static_cast<uint16_t>(upper);
}

// Round-to-nearest-even of an fp64 value to bfloat16, rounding once: the fp32
// conversion can land exactly on a bfloat16 midpoint that the fp64 value is
// not on; the value is then moved one fp32 step toward the fp64 value, so the
// bfloat16 rounding sees which side of the midpoint it lies.
uint16_t double_to_bf16_bits(double x) {
  float f = static_cast<float>(x);
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0xffffu) == 0x8000u && static_cast<double>(f) != x && std::isfinite(f)) {
    if (std::fabs(x) > std::fabs(static_cast<double>(f)))
      u += 1;
    else
      u -= 1;
    std::memcpy(&f, &u, 4);
  }
  return float_to_bf16_bits(f);
}

float load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == DT_BF16) return bf16_bits_to_float(static_cast<const uint16_t*>(base)[i]);
  return static_cast<const float*>(base)[i];
}

void store_elem(void* base, int dtype, int64_t i, float v) {
  if (dtype == DT_BF16)
    static_cast<uint16_t*>(base)[i] = float_to_bf16_bits(v);
  else
    static_cast<float*>(base)[i] = v;
}

// Index of the largest value among the entries whose `eligible` flag is set
// and that are not yet `taken`; strict ">" keeps the lower index on ties.
template <typename V>
int pick_largest(const std::vector<V>& value, const std::vector<char>& eligible,
                 const std::vector<char>& taken) {
  int best = -1;
  for (size_t i = 0; i < value.size(); ++i) {
    if (!eligible[i] || taken[i]) continue;
    if (best < 0 || value[i] > value[static_cast<size_t>(best)]) best = static_cast<int>(i);
  }
  return best;
}

}  // namespace

extern "C" {

// Softmax top-K routing (router "probabilities" whose top-k indices and
// scores feed dispatch; [AutoEP-prep] "Testing Done": exact routes,
// routing-score gradients).
//   logits [T,E] fp32 -> idx [T,K] int32 (descending key, ties lower index),
//   w [T,K] fp32.
// renorm = 1: w_k = p_k / sum_{j in top-K} p_j, which equals
//   exp(l_k - l_max) / sum_{j in top-K} exp(l_j - l_max) (the full softmax
//   denominator cancels).  renorm = 0: w_k = softmax(l)_k over all E.
// The weights are multiplied by route_scale, all in fp64, then rounded to fp32.
// Returns 0, or -1 for invalid sizes.
int orc_route_softmax(const float* logits, int64_t T, int E, int K, int renorm,
                      double route_scale, int32_t* idx, float* w) {
  if (T < 0 || E <= 0 || K <= 0 || K > E) return -1;
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::vector<float> key(l, l + E);
    std::vector<char> eligible(static_cast<size_t>(E), 1), taken(static_cast<size_t>(E), 0);
    for (int k = 0; k < K; ++k) {
      int e = pick_largest(key, eligible, taken);
      taken[static_cast<size_t>(e)] = 1;
      idx[t * K + k] = e;
    }
    const double l_max = static_cast<double>(l[idx[t * K]]);
    double den = 0.0;
    if (renorm) {
      for (int k = 0; k < K; ++k) den += std::exp(static_cast<double>(l[idx[t * K + k]]) - l_max);
    } else {
      for (int e = 0; e < E; ++e) den += std::exp(static_cast<double>(l[e]) - l_max);
    }
    for (int k = 0; k < K; ++k) {
      double p = std::exp(static_cast<double>(l[idx[t * K + k]]) - l_max) / den;
      w[t * K + k] = static_cast<float>(p * route_scale);
    }
  }
  return 0;
}

// Group-limited sigmoid routing with a score-correction bias ([AutoEP-prep]
// "Testing Done" names the score-correction bias; the algorithm is the
// reading stated at the top of this file).
//   s_e   = 1 / (1 + exp(-l_e))                       (fp64)
//   key_e = s_e + bias_e                              (fp64; bias may be NULL)
//   experts are split into n_groups contiguous groups of E / n_groups;
//   group score = sum of the group's top `group_score_topk` keys, added in
//   descending order;
//   keep the top `topk_groups` groups, then the top-K experts by key among
//   them (descending key, ties lower index);
//   w_k = s_k / sum_j s_j (renorm = 1) or s_k (renorm = 0), times route_scale,
//   in fp64, rounded to fp32.
int orc_route_sigmoid_grouped(const float* logits, const float* bias, int64_t T, int E, int K,
                              int n_groups, int topk_groups, int group_score_topk, int renorm,
                              double route_scale, int32_t* idx, float* w) {
  if (T < 0 || E <= 0 || K <= 0 || n_groups <= 0 || E % n_groups) return -1;
  const int gsz = E / n_groups;
  if (topk_groups <= 0 || topk_groups > n_groups || group_score_topk <= 0 ||
      group_score_topk > gsz || K > topk_groups * gsz)
    return -1;
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    std::vector<double> s(static_cast<size_t>(E)), key(static_cast<size_t>(E));
    for (int e = 0; e < E; ++e) {
      s[static_cast<size_t>(e)] = 1.0 / (1.0 + std::exp(-static_cast<double>(l[e])));
      key[static_cast<size_t>(e)] = s[static_cast<size_t>(e)] + (bias ? static_cast<double>(bias[e]) : 0.0);
    }
    std::vector<double> gscore(static_cast<size_t>(n_groups));
    for (int g = 0; g < n_groups; ++g) {
      std::vector<double> gkey(key.begin() + g * gsz, key.begin() + (g + 1) * gsz);
      std::vector<char> all(static_cast<size_t>(gsz), 1), taken(static_cast<size_t>(gsz), 0);
      double sum = 0.0;
      for (int j = 0; j < group_score_topk; ++j) {
        int i = pick_largest(gkey, all, taken);
        taken[static_cast<size_t>(i)] = 1;
        sum += gkey[static_cast<size_t>(i)];
      }
      gscore[static_cast<size_t>(g)] = sum;
    }
    std::vector<char> gall(static_cast<size_t>(n_groups), 1), gkeep(static_cast<size_t>(n_groups), 0);
    for (int j = 0; j < topk_groups; ++j) gkeep[static_cast<size_t>(pick_largest(gscore, gall, gkeep))] = 1;
    std::vector<char> eligible(static_cast<size_t>(E)), taken(static_cast<size_t>(E), 0);
    for (int e = 0; e < E; ++e) eligible[static_cast<size_t>(e)] = gkeep[static_cast<size_t>(e / gsz)];
    for (int k = 0; k < K; ++k) {
      int e = pick_largest(key, eligible, taken);
      taken[static_cast<size_t>(e)] = 1;
      idx[t * K + k] = e;
    }
    double den = 0.0;
    for (int k = 0; k < K; ++k) den += s[static_cast<size_t>(idx[t * K + k])];
    for (int k = 0; k < K; ++k) {
      double sk = s[static_cast<size_t>(idx[t * K + k])];
      double p = renorm ? sk / den : sk;
      w[t * K + k] = static_cast<float>(p * route_scale);
    }
  }
  return 0;
}

// Dispatch layout ([AutoEP-DeepEP] "Why": a token is sent once per
// destination rank rather than once per selected expert, and arrivals are
// grouped by expert for the grouped GEMM; [AutoEP-prep] "Summary": no
// split-count all-to-all and no device-to-host split materialisation).
// Destination ranks are virtual: rank(e) = e / (E / R).
//   cnt_e[E], off_e[E+1]           per-expert counts and exclusive offsets
//   pos[t,k] = off_e[e] + #{t' < t : e in idx[t']}           (-1 if dropped)
//   recv_token[pos] = t, recv_k[pos] = k                     ([T*K], tail -1)
//   cnt_send_r[r] = #{t : r in ranks(t)}, off_send_r[R+1], S = off_send_r[R]
//   send row of (t, r) = off_send_r[r] + #{t' < t : r in ranks(t')}
//   send_token[row] = t                                      ([T*min(K,R)], tail -1)
//   send_row_of[t,k] = send row of (t, rank(idx[t,k]))        (-1 if dropped)
//   recv_send_row[pos[t,k]] = send_row_of[t,k]               (tail -1)
//   cnt_recv_r[r] = sum of cnt_e over r's experts, off_recv_r[r] = off_e[r*E/R]
// Returns the number of dropped entries, or -1 for invalid sizes.
//
// Padded layout (align > 1; the TorchAO padded permute of [Titan-absorb]
// "Implementation", zero-sentinel scores): every expert segment is rounded up
// to a multiple of `align` rows, off_e[e+1] = off_e[e] + ceil(cnt_e/align)*align;
// the pad rows carry recv_token = recv_k = recv_send_row = -1, and the
// receive arrays hold T*K + E*(align-1) rows.  align = 1: no padding.
int64_t orc_layout(const int32_t* idx, int64_t T, int K, int E, int R, int align, int32_t* cnt_e,
                   int32_t* off_e, int32_t* cnt_send_r, int32_t* off_send_r, int32_t* cnt_recv_r,
                   int32_t* off_recv_r, int32_t* pos, int32_t* recv_token, int32_t* recv_k,
                   int32_t* send_token, int32_t* send_row_of, int32_t* recv_send_row,
                   int64_t* S_out) {
  if (T < 0 || K <= 0 || E <= 0 || R <= 0 || E % R || align < 1) return -1;
  const int epr = E / R;
  const int64_t send_cap = T * (K < R ? K : R);
  const int64_t recv_cap = T * K + static_cast<int64_t>(E) * (align - 1);
  int64_t dropped = 0;

  std::vector<char> valid(static_cast<size_t>(T * K), 0);
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int32_t e = idx[t * K + k];
      bool ok = e >= 0 && e < E;
      for (int j = 0; j < k && ok; ++j)
        if (valid[static_cast<size_t>(t * K + j)] && idx[t * K + j] == e) ok = false;
      valid[static_cast<size_t>(t * K + k)] = ok ? 1 : 0;
      if (!ok) ++dropped;
    }

  for (int e = 0; e < E; ++e) cnt_e[e] = 0;
  for (int64_t i = 0; i < T * K; ++i)
    if (valid[static_cast<size_t>(i)]) ++cnt_e[idx[i]];
  off_e[0] = 0;
  for (int e = 0; e < E; ++e) off_e[e + 1] = off_e[e] + (cnt_e[e] + align - 1) / align * align;

  std::vector<int64_t> seen_e(static_cast<size_t>(E), 0);
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t i = t * K + k;
      if (!valid[static_cast<size_t>(i)]) {
        pos[i] = -1;
        continue;
      }
      int e = idx[i];
      int64_t p = off_e[e] + seen_e[static_cast<size_t>(e)]++;
      pos[i] = static_cast<int32_t>(p);
      recv_token[p] = static_cast<int32_t>(t);
      recv_k[p] = k;
    }
  for (int e = 0; e < E; ++e)  // pad rows of each segment
    for (int64_t p = off_e[e] + cnt_e[e]; p < off_e[e + 1]; ++p)
      recv_token[p] = recv_k[p] = recv_send_row[p] = -1;
  for (int64_t p = off_e[E]; p < recv_cap; ++p) recv_token[p] = recv_k[p] = recv_send_row[p] = -1;

  // ranks(t): the set of destination ranks of token t's valid entries
  std::vector<char> in_ranks(static_cast<size_t>(R));
  for (int r = 0; r < R; ++r) cnt_send_r[r] = 0;
  for (int64_t t = 0; t < T; ++t) {
    std::fill(in_ranks.begin(), in_ranks.end(), 0);
    for (int k = 0; k < K; ++k)
      if (valid[static_cast<size_t>(t * K + k)]) in_ranks[static_cast<size_t>(idx[t * K + k] / epr)] = 1;
    for (int r = 0; r < R; ++r) cnt_send_r[r] += in_ranks[static_cast<size_t>(r)];
  }
  off_send_r[0] = 0;
  for (int r = 0; r < R; ++r) off_send_r[r + 1] = off_send_r[r] + cnt_send_r[r];
  const int64_t S = off_send_r[R];

  std::vector<int64_t> seen_r(static_cast<size_t>(R), 0);
  std::vector<int64_t> row_of_rank(static_cast<size_t>(R));
  for (int64_t t = 0; t < T; ++t) {
    std::fill(in_ranks.begin(), in_ranks.end(), 0);
    for (int k = 0; k < K; ++k)
      if (valid[static_cast<size_t>(t * K + k)]) in_ranks[static_cast<size_t>(idx[t * K + k] / epr)] = 1;
    for (int r = 0; r < R; ++r) {
      row_of_rank[static_cast<size_t>(r)] = -1;
      if (!in_ranks[static_cast<size_t>(r)]) continue;
      int64_t row = off_send_r[r] + seen_r[static_cast<size_t>(r)]++;
      row_of_rank[static_cast<size_t>(r)] = row;
      send_token[row] = static_cast<int32_t>(t);
    }
    for (int k = 0; k < K; ++k) {
      int64_t i = t * K + k;
      if (!valid[static_cast<size_t>(i)]) {
        send_row_of[i] = -1;
        continue;
      }
      int64_t row = row_of_rank[static_cast<size_t>(idx[i] / epr)];
      send_row_of[i] = static_cast<int32_t>(row);
      recv_send_row[pos[i]] = static_cast<int32_t>(row);
    }
  }
  for (int64_t row = S; row < send_cap; ++row) send_token[row] = -1;

  for (int r = 0; r < R; ++r) {
    cnt_recv_r[r] = 0;
    for (int e = r * epr; e < (r + 1) * epr; ++e) cnt_recv_r[r] += cnt_e[e];
    off_recv_r[r] = off_e[r * epr];
  }
  off_recv_r[R] = off_e[E];
  *S_out = S;
  return dropped;
}

// Dispatch ([AutoEP-DeepEP] "Why": DeepEP takes tokens before top-k
// expansion and replicates them itself; [Titan-absorb] "Implementation": the
// per-row router scores are gathered expert-major with the same permutation
// and returned as routed_scores_R).
//   recv[pos[t,k]] = x[t]            (bit copy of a row of row_bytes bytes)
//   recv_w[pos[t,k]] = w[t,k]        (if recv_w is not NULL)
//   send[send_row_of[t,k]] = x[t]    (if send is not NULL)
void orc_dispatch(const void* x, int64_t row_bytes, int64_t T, int K, const int32_t* pos,
                  const float* w, const int32_t* send_row_of, void* recv, float* recv_w,
                  void* send) {
  const char* src = static_cast<const char*>(x);
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t p = pos[t * K + k];
      if (p < 0) continue;
      std::memcpy(static_cast<char*>(recv) + p * row_bytes, src + t * row_bytes,
                  static_cast<size_t>(row_bytes));
      if (recv_w) recv_w[p] = w[t * K + k];
      if (send) {
        int64_t s = send_row_of[t * K + k];
        std::memcpy(static_cast<char*>(send) + s * row_bytes, src + t * row_bytes,
                    static_cast<size_t>(row_bytes));
      }
    }
}

// Combine ([AutoEP-DeepEP] "Why": DeepEP reduces the weighted sum in its
// combine, restoring token order; [Titan-absorb] "Motivation": with the
// router scores absorbed into the W2 input the combine is a plain sum).
//   out[t,h] = round( fp32 sum over k, in k order, of w[t,k] * y[pos[t,k],h] )
// with acc = fma(w, y, acc) starting from +0 (w == NULL: acc = acc + y).
// The sum is rounded once to the row dtype (bf16 round-to-nearest-even).
void orc_combine(const void* y, int dtype, int64_t H, int64_t T, int K, const int32_t* pos,
                 const float* w, void* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        int64_t p = pos[t * K + k];
        if (p < 0) continue;
        float v = load_elem(y, dtype, p * H + h);
        acc = w ? std::fma(w[t * K + k], v, acc) : acc + v;
      }
      store_elem(out, dtype, t * H + h, acc);
    }
}

// Combine backward ([AutoEP-DeepEP] "Why" and the review-fix commit: the
// gradient of a combine is a dispatch replayed against the forward handle,
// and the backward must also return the router-score gradient).
//   gy[pos[t,k],h] = round(w[t,k] * g[t,h])   (fp32 product, then the dtype)
//   gy[pos[t,k],h] = g[t,h]                   (w == NULL: plain sum)
//   gw[t,k] = sum_h g[t,h] * y[pos[t,k],h]     (fp64; only if w and gw given;
//                                              0 for a dropped entry)
void orc_combine_bwd(const void* g, const void* y, int dtype, int64_t H, int64_t T, int K,
                     const int32_t* pos, const float* w, void* gy, double* gw) {
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t p = pos[t * K + k];
      if (p < 0) {
        if (w && gw) gw[t * K + k] = 0.0;
        continue;
      }
      double dot = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        float gv = load_elem(g, dtype, t * H + h);
        if (w && gw) dot += static_cast<double>(gv) * static_cast<double>(load_elem(y, dtype, p * H + h));
        store_elem(gy, dtype, p * H + h, w ? w[t * K + k] * gv : gv);
      }
      if (w && gw) gw[t * K + k] = dot;
    }
}

// Dispatch backward ([AutoEP-DeepEP] "Why": the gradient of a dispatch is a
// combine replayed against the forward handle), with unit weights:
//   gx[t,h] = round( fp32 sum over k, in k order, of grecv[pos[t,k],h] )
void orc_dispatch_bwd(const void* grecv, int dtype, int64_t H, int64_t T, int K,
                      const int32_t* pos, void* gx) {
  orc_combine(grecv, dtype, H, T, K, pos, nullptr, gx);
}

// Router-score absorption, forward ([Titan-absorb] "Implementation":
// GroupedLinear scales the W2 input in float32 and restores the input dtype
// before the grouped GEMM):
//   hs[r,i] = round(h[r,i] * recv_w[r])   for r < rows
void orc_scale_rows(const void* h, int dtype, int64_t I, int64_t rows, const float* recv_w,
                    void* hs) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < I; ++i)
      store_elem(hs, dtype, r * I + i, load_elem(h, dtype, r * I + i) * recv_w[r]);
}

// Router-score absorption, backward (the same linear scaling; the score
// gradient is the dot product of the incoming gradient with the unscaled
// input row):
//   gh[r,i]  = round(recv_w[r] * ghs[r,i])            for r < rows
//   gw[t,k]  = sum_i ghs[pos[t,k],i] * h[pos[t,k],i]  (fp64; 0 if dropped)
void orc_scale_rows_bwd(const void* ghs, const void* h, int dtype, int64_t I, int64_t rows,
                        int64_t T, int K, const int32_t* pos, const float* recv_w, void* gh,
                        double* gw) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < I; ++i)
      store_elem(gh, dtype, r * I + i, recv_w[r] * load_elem(ghs, dtype, r * I + i));
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t p = pos[t * K + k];
      double dot = 0.0;
      if (p >= 0)
        for (int64_t i = 0; i < I; ++i)
          dot += static_cast<double>(load_elem(ghs, dtype, p * I + i)) *
                 static_cast<double>(load_elem(h, dtype, p * I + i));
      gw[t * K + k] = dot;
    }
}

// fp64 weighted combine, the exact definition without intermediate rounding:
//   out[t,h] = sum_k w[t,k] * y[pos[t,k],h]   (w == NULL: unit weights)
// Used by the pins (adjoint identities, absorption equivalence) and as the
// yardstick for the fp32-accumulated combine.
void orc_combine_f64(const double* y, int64_t H, int64_t T, int K, const int32_t* pos,
                     const double* w, double* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        int64_t p = pos[t * K + k];
        if (p < 0) continue;
        acc += (w ? w[t * K + k] : 1.0) * y[p * H + h];
      }
      out[t * H + h] = acc;
    }
}

// fp64 dispatch: recv[pos[t,k]] = x[t] (used by the adjoint pins).
void orc_dispatch_f64(const double* x, int64_t H, int64_t T, int K, const int32_t* pos,
                      double* recv) {
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int64_t p = pos[t * K + k];
      if (p < 0) continue;
      for (int64_t h = 0; h < H; ++h) recv[p * H + h] = x[t * H + h];
    }
}

// fp32 -> bf16 round-to-nearest-even, exported so that the tests can round
// reference values the same way the definitions above do.
void orc_f32_to_bf16(const float* src, int64_t n, uint16_t* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = float_to_bf16_bits(src[i]);
}

// Router backward to the logits (the router-score and router-parameter
// gradients of [AutoEP-prep] "Testing Done"; dL/dw is the router-score
// gradient that the combine backward returns).  The selection is fixed; the
// weights as functions of the logits are
//   softmax, renorm:     w_k = c * q_k,  q_k = exp(l_k) / sum_{j in sel} exp(l_j)
//   softmax, no renorm:  w_k = c * p_k,  p = softmax(l) over all E
//   sigmoid, renorm:     w_k = c * s_k / S,  s = sigmoid(l), S = sum_{j in sel} s_j
//   sigmoid, no renorm:  w_k = c * s_k
// (c = route_scale; the correction bias enters only the selection and gets no
// gradient).  Their derivatives, in fp64:
//   softmax renorm:     dL/dl_j = c q_j (gw_j - sum_k q_k gw_k),  j selected; 0 else
//   softmax no renorm:  dL/dl_e = c p_e (gw_e - sum_k p_k gw_k),  gw_e = 0 if e not selected
//   sigmoid renorm:     dL/dl_j = s_j (1 - s_j) (c / S) (gw_j - sum_k gw_k s_k / S)
//   sigmoid no renorm:  dL/dl_j = c gw_j s_j (1 - s_j)
// glogits [T,E] fp64 (every entry written).
int orc_route_bwd(const float* logits, int64_t T, int E, int K, int score_fn, int renorm,
                  double route_scale, const int32_t* idx, const double* gw, double* glogits) {
  if (T < 0 || E <= 0 || K <= 0 || K > E) return -1;
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    const int32_t* sel = idx + t * K;
    const double* g = gw + t * K;
    double* out = glogits + t * E;
    for (int e = 0; e < E; ++e) out[e] = 0.0;
    if (score_fn == 0) {  // softmax
      const double l_max = static_cast<double>(l[sel[0]]);
      double den = 0.0;
      if (renorm) {
        for (int k = 0; k < K; ++k) den += std::exp(static_cast<double>(l[sel[k]]) - l_max);
        double dot = 0.0;
        for (int k = 0; k < K; ++k)
          dot += std::exp(static_cast<double>(l[sel[k]]) - l_max) / den * g[k];
        for (int k = 0; k < K; ++k) {
          double q = std::exp(static_cast<double>(l[sel[k]]) - l_max) / den;
          out[sel[k]] = route_scale * q * (g[k] - dot);
        }
      } else {
        double m = static_cast<double>(l[0]);
        for (int e = 1; e < E; ++e) m = std::max(m, static_cast<double>(l[e]));
        for (int e = 0; e < E; ++e) den += std::exp(static_cast<double>(l[e]) - m);
        std::vector<double> gfull(static_cast<size_t>(E), 0.0);
        for (int k = 0; k < K; ++k) gfull[static_cast<size_t>(sel[k])] = g[k];
        double dot = 0.0;
        for (int k = 0; k < K; ++k)
          dot += std::exp(static_cast<double>(l[sel[k]]) - m) / den * g[k];
        for (int e = 0; e < E; ++e) {
          double p = std::exp(static_cast<double>(l[e]) - m) / den;
          out[e] = route_scale * p * (gfull[static_cast<size_t>(e)] - dot);
        }
      }
    } else {  // sigmoid
      std::vector<double> s(static_cast<size_t>(K));
      double S = 0.0;
      for (int k = 0; k < K; ++k) {
        s[static_cast<size_t>(k)] = 1.0 / (1.0 + std::exp(-static_cast<double>(l[sel[k]])));
        S += s[static_cast<size_t>(k)];
      }
      if (renorm) {
        double dot = 0.0;
        for (int k = 0; k < K; ++k) dot += g[k] * s[static_cast<size_t>(k)] / S;
        for (int k = 0; k < K; ++k) {
          double sk = s[static_cast<size_t>(k)];
          out[sel[k]] = sk * (1.0 - sk) * (route_scale / S) * (g[k] - dot);
        }
      } else {
        for (int k = 0; k < K; ++k) {
          double sk = s[static_cast<size_t>(k)];
          out[sel[k]] = route_scale * g[k] * sk * (1.0 - sk);
        }
      }
    }
  }
  return 0;
}

// Staged (wire-faithful) dispatch and combine ([AutoEP-DeepEP] "Why": a
// token goes to each destination rank once, not once per selected expert;
// the receiving side groups the arrivals by expert, and the combine returns
// one reduced row per (token, rank)).  The send rows come from orc_dispatch
// with `send`; then:
//
// expand: the receiving side copies each arrived row to the rows of its
// experts on that rank:  recv[pos[t,k]] = send[send_row_of[t,k]].
void orc_expand(const void* send, int64_t row_bytes, int64_t T, int K, const int32_t* pos,
                const int32_t* send_row_of, void* recv) {
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      const int64_t p = pos[t * K + k];
      if (p < 0) continue;
      std::memcpy(static_cast<char*>(recv) + p * row_bytes,
                  static_cast<const char*>(send) + static_cast<int64_t>(send_row_of[t * K + k]) * row_bytes,
                  static_cast<size_t>(row_bytes));
    }
}

// combine, stage 1 (on the expert side): one partial row per send row s of
// token t, the fp32 sum in k order of w[t,k] * y[pos[t,k]] over the entries k
// with send_row_of[t,k] == s (fma; acc + y when w is NULL), rounded once to
// the row dtype (what travels back).
void orc_combine_partial(const void* y, int dtype, int64_t H, int64_t T, int K,
                         const int32_t* pos, const int32_t* send_row_of, const float* w,
                         void* partial) {
  for (int64_t t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      const int32_t s = send_row_of[t * K + k];
      if (s < 0) continue;
      bool first = true;
      for (int j = 0; j < k; ++j)
        if (send_row_of[t * K + j] == s) first = false;
      if (!first) continue;
      for (int64_t h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int j = k; j < K; ++j) {
          if (send_row_of[t * K + j] != s) continue;
          const float v = load_elem(y, dtype, static_cast<int64_t>(pos[t * K + j]) * H + h);
          acc = w ? std::fma(w[t * K + j], v, acc) : acc + v;
        }
        store_elem(partial, dtype, static_cast<int64_t>(s) * H + h, acc);
      }
    }
}

// combine, stage 2 (back on the token's side): the fp32 sum of the token's
// partial rows, each distinct send row once, in the order its first entry
// appears in k, rounded once.
void orc_combine_reduce(const void* partial, int dtype, int64_t H, int64_t T, int K,
                        const int32_t* send_row_of, void* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        const int32_t s = send_row_of[t * K + k];
        if (s < 0) continue;
        bool first = true;
        for (int j = 0; j < k; ++j)
          if (send_row_of[t * K + j] == s) first = false;
        if (first) acc = acc + load_elem(partial, dtype, static_cast<int64_t>(s) * H + h);
      }
      store_elem(out, dtype, t * H + h, acc);
    }
}

// Router-score absorption fused with the W2 projection ([Titan-absorb]
// "Implementation": GroupedLinear scales the W2 input by the routed score in
// float32 and restores the input dtype before the grouped GEMM, so the W2 GEMM
// of expert e consumes the scaled rows of e's receive segment):
//   e(r)    = the expert whose receive segment [off_e[e], off_e[e+1]) holds r
//   hs[r,i] = round_bf16(h[r,i] * recv_w[r])                     (fp32 product)
//   y[r,n]  = round_bf16(sum_i hs[r,i] * W2[e(r)][n,i])   (fp64 sum, one rounding)
// for the real rows of a segment (r - off_e[e] < cnt_e[e]); a pad row of a
// padded layout, or a row outside every segment, is 0.  W2 is stored
// [E][H][I]: output column n of expert e is the I-vector W2[e][n].  Only the
// listed rows are computed: y and y64 are [nrows, H].
void orc_w2_absorbed(const uint16_t* h, int64_t I, const float* recv_w, const uint16_t* w2,
                     int64_t H, int E, const int32_t* off_e, const int32_t* cnt_e,
                     const int64_t* rows, int64_t nrows, uint16_t* y, double* y64) {
  std::vector<double> hs(static_cast<size_t>(I));
  for (int64_t j = 0; j < nrows; ++j) {
    const int64_t r = rows[j];
    int e = -1;
    for (int c = 0; c < E; ++c)
      if (r >= off_e[c] && r < off_e[c + 1]) e = c;
    const bool real = e >= 0 && r - off_e[e] < cnt_e[e];
    if (real)
      for (int64_t i = 0; i < I; ++i) {
        const float scaled = bf16_bits_to_float(h[r * I + i]) * recv_w[r];
        hs[i] = bf16_bits_to_float(float_to_bf16_bits(scaled));
      }
    for (int64_t n = 0; n < H; ++n) {
      double acc = 0.0;
      if (real) {
        const uint16_t* wrow = w2 + (static_cast<int64_t>(e) * H + n) * I;
        for (int64_t i = 0; i < I; ++i) acc += hs[i] * static_cast<double>(bf16_bits_to_float(wrow[i]));
      }
      y64[j * H + n] = acc;
      y[j * H + n] = double_to_bf16_bits(acc);
    }
  }
}

// fp64 -> bfloat16 round-to-nearest-even of n values (for the tests' pins).
void orc_f64_to_bf16(const double* src, int64_t n, uint16_t* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = double_to_bf16_bits(src[i]);
}

}  // extern "C"
