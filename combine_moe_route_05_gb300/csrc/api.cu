// C ABI of the MoE routing library: argument validation, the handle and its
// workspace plan, and the launches.  Every check that can be made on the host
// is made here, before anything is launched; a failed check launches nothing.
#include <cmath>
#include <cstdint>
#include <new>

#include "internal.h"

namespace moe {
size_t layout_smem_bytes(int E, int R);
cudaError_t prepare_layout_kernels();
}  // namespace moe

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool config_valid(const moe_config* c) {
  if (!c) return false;
  const int E = c->num_experts, K = c->top_k, R = c->num_ranks, G = c->num_groups;
  if (E < 1 || E > MOE_MAX_EXPERTS) return false;
  if (K < 1 || K > MOE_MAX_TOPK || K > E) return false;
  if (R < 1 || E % R != 0) return false;
  if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID) return false;
  if (G < 1 || G > 32 || E % G != 0) return false;
  if (G > 1 && c->score_fn != MOE_SCORE_SIGMOID) return false;
  if (c->topk_groups < 1 || c->topk_groups > G) return false;
  if (c->group_score_topk < 1 || c->group_score_topk > E / G) return false;
  if (K > c->topk_groups * (E / G)) return false;
  if (c->renorm != 0 && c->renorm != 1) return false;
  if (!std::isfinite(c->route_scale)) return false;
  if (c->max_tokens < 0) return false;
  if (c->pad_align < 0 || c->pad_align > 4096) return false;
  const int64_t pad = c->pad_align > 1 ? c->pad_align : 1;
  if (static_cast<int64_t>(c->max_tokens) * K + static_cast<int64_t>(E) * (pad - 1) > INT32_MAX)
    return false;
  return true;
}

struct Plan {
  size_t flags, ticket, cnt_e, off_e, cnt_send_r, off_send_r, cnt_recv_r, off_recv_r, S;
  size_t pos, recv_token, recv_k, send_token, send_row_of, recv_send_row, tile_hist, total;
  int max_tiles;
};

Plan plan(const moe_config* c) {
  Plan p{};
  const size_t E = c->num_experts, R = c->num_ranks, K = c->top_k;
  const size_t T = c->max_tokens;
  const size_t i4 = sizeof(int32_t);
  p.max_tiles = static_cast<int>(T > 0 ? (T + MOE_LAYOUT_TILE_TOKENS - 1) / MOE_LAYOUT_TILE_TOKENS : 1);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + (bytes ? bytes : 1));
    return at;
  };
  p.flags = take(i4);
  p.ticket = take(sizeof(uint64_t));
  p.cnt_e = take(E * i4);
  p.off_e = take((E + 1) * i4);
  p.cnt_send_r = take(R * i4);
  p.off_send_r = take((R + 1) * i4);
  p.cnt_recv_r = take(R * i4);
  p.off_recv_r = take((R + 1) * i4);
  p.S = take(i4);
  const size_t RR = T * K + E * static_cast<size_t>(c->pad_align > 1 ? c->pad_align - 1 : 0);
  p.pos = take(T * K * i4);
  p.recv_token = take(RR * i4);
  p.recv_k = take(RR * i4);
  p.send_token = take(T * (K < R ? K : R) * i4);
  p.send_row_of = take(T * K * i4);
  p.recv_send_row = take(RR * i4);
  p.tile_hist = take((E + R) * static_cast<size_t>(p.max_tiles) * i4);
  p.total = o;
  return p;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_dtype(int32_t d) { return d == MOE_BF16 || d == MOE_F32; }

int64_t elt_bytes(int32_t d) { return d == MOE_BF16 ? 2 : 4; }

// A row tensor argument: non-null, 16-byte aligned, row size a multiple of 16.
bool row_ok(const void* p, int32_t width, int32_t dtype) {
  if (!p || width <= 0 || !valid_dtype(dtype)) return false;
  if (!aligned(p, 16)) return false;
  return (static_cast<int64_t>(width) * elt_bytes(dtype)) % 16 == 0;
}

// With an empty layout (T = 0) the row tensors are empty and may be null:
// nothing is launched, only the width and dtype are checked.
bool empty_rows_ok(int32_t width, int32_t dtype) {
  return width > 0 && valid_dtype(dtype) && (static_cast<int64_t>(width) * elt_bytes(dtype)) % 16 == 0;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Every launch goes to the current device, and every pointer a call gets must
// live on the handle's device: a call made while another device is current
// is refused before anything is launched.
bool on_handle_device(const moe_handle* h) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == h->device;
}

}  // namespace

namespace moe {
bool valid_config(const moe_config* c) { return config_valid(c); }
}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID: return "MOE_ERR_INVALID: invalid argument or configuration";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY: more tokens than the handle's max_tokens";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_STATE: return "MOE_ERR_STATE: no dispatch layout on this handle yet";
  }
  return "unknown moe_status";
}

size_t moe_workspace_bytes(const moe_config* c) {
  if (!config_valid(c)) return 0;
  return plan(c).total;
}

moe_status moe_handle_create(const moe_config* c, void* d_workspace, size_t workspace_bytes,
                             moe_handle** out) {
  if (!out) return MOE_ERR_INVALID;
  *out = nullptr;
  if (!config_valid(c) || !d_workspace || !aligned(d_workspace, kAlign)) return MOE_ERR_INVALID;
  const Plan p = plan(c);
  if (workspace_bytes < p.total) return MOE_ERR_INVALID;
  if (moe::layout_smem_bytes(c->num_experts, c->num_ranks) > 227 * 1024) return MOE_ERR_INVALID;

  int dev = 0, sms = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  // fails with "no kernel image" on a device the library was not built for
  if (moe::prepare_layout_kernels() != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::prepare_w2_kernel() != cudaSuccess) return MOE_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  if (cudaMemset(ws, 0, p.S + sizeof(int32_t)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;

  moe_handle* h = new (std::nothrow) moe_handle;
  if (!h) return MOE_ERR_INVALID;
  h->cfg = *c;
  h->device = dev;
  h->num_sms = sms;
  h->l2_bytes = l2;
  h->T = -1;
  h->max_tiles = p.max_tiles;
  h->pad = c->pad_align > 1 ? c->pad_align : 1;
  h->wait_ns = MOE_DEFAULT_WAIT_LIMIT_NS;
  h->flags = reinterpret_cast<uint32_t*>(ws + p.flags);
  h->ticket = reinterpret_cast<uint32_t*>(ws + p.ticket);
  h->cnt_e = reinterpret_cast<int32_t*>(ws + p.cnt_e);
  h->off_e = reinterpret_cast<int32_t*>(ws + p.off_e);
  h->cnt_send_r = reinterpret_cast<int32_t*>(ws + p.cnt_send_r);
  h->off_send_r = reinterpret_cast<int32_t*>(ws + p.off_send_r);
  h->cnt_recv_r = reinterpret_cast<int32_t*>(ws + p.cnt_recv_r);
  h->off_recv_r = reinterpret_cast<int32_t*>(ws + p.off_recv_r);
  h->S = reinterpret_cast<int32_t*>(ws + p.S);
  h->pos = reinterpret_cast<int32_t*>(ws + p.pos);
  h->recv_token = reinterpret_cast<int32_t*>(ws + p.recv_token);
  h->recv_k = reinterpret_cast<int32_t*>(ws + p.recv_k);
  h->send_token = reinterpret_cast<int32_t*>(ws + p.send_token);
  h->send_row_of = reinterpret_cast<int32_t*>(ws + p.send_row_of);
  h->recv_send_row = reinterpret_cast<int32_t*>(ws + p.recv_send_row);
  h->tile_hist = reinterpret_cast<int32_t*>(ws + p.tile_hist);
  *out = h;
  return MOE_OK;
}

moe_status moe_handle_destroy(moe_handle* h) {
  if (!h) return MOE_ERR_INVALID;
  delete h;
  return MOE_OK;
}

moe_status moe_route_topk(moe_handle* h, const float* d_logits, const float* d_bias, int32_t T,
                          int32_t* d_idx, float* d_w, void* stream) {
  if (!h || T < 0) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (T > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (T > 0 && (!d_logits || !d_idx || !d_w)) return MOE_ERR_INVALID;
  if (!aligned(d_logits, 4) || !aligned(d_idx, 4) || !aligned(d_w, 4) || !aligned(d_bias, 4))
    return MOE_ERR_INVALID;
  if (d_bias && h->cfg.score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_route_topk(h, d_logits, d_bias, T, d_idx, d_w, as_stream(stream)));
}

moe_status moe_route_bwd(const moe_handle* h, const float* d_logits, const int32_t* d_idx,
                         const float* d_gw, int32_t T, float* d_glogits, void* stream) {
  if (!h || T < 0) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (T > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (T > 0 && (!d_logits || !d_idx || !d_gw || !d_glogits)) return MOE_ERR_INVALID;
  if (!aligned(d_logits, 4) || !aligned(d_idx, 4) || !aligned(d_gw, 4) || !aligned(d_glogits, 4))
    return MOE_ERR_INVALID;
  return from_cuda(
      moe::launch_route_bwd(h, d_logits, d_idx, d_gw, T, d_glogits, as_stream(stream)));
}

moe_status moe_dispatch_layout(moe_handle* h, const int32_t* d_idx, int32_t T, void* stream) {
  if (!h || T < 0) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (T > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  if (T > 0 && (!d_idx || !aligned(d_idx, 4))) return MOE_ERR_INVALID;
  const moe_status st = from_cuda(moe::launch_layout(h, d_idx, T, as_stream(stream)));
  if (st == MOE_OK) h->T = T;
  return st;
}

moe_status moe_layout_view(const moe_handle* h, moe_layout* out) {
  if (!h || !out) return MOE_ERR_INVALID;
  out->cnt_e = h->cnt_e;
  out->off_e = h->off_e;
  out->cnt_send_r = h->cnt_send_r;
  out->off_send_r = h->off_send_r;
  out->cnt_recv_r = h->cnt_recv_r;
  out->off_recv_r = h->off_recv_r;
  out->pos = h->pos;
  out->recv_token = h->recv_token;
  out->recv_k = h->recv_k;
  out->send_token = h->send_token;
  out->send_row_of = h->send_row_of;
  out->recv_send_row = h->recv_send_row;
  out->S = h->S;
  out->num_tokens = h->T;
  out->pad_align = h->pad;
  return MOE_OK;
}

moe_status moe_dispatch(const moe_handle* h, const void* d_x, int32_t H, int32_t dtype,
                        const float* d_w, void* d_recv, float* d_recv_w, void* d_send,
                        void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_x, H, dtype) || !row_ok(d_recv, H, dtype)) return MOE_ERR_INVALID;
  if (d_send && !row_ok(d_send, H, dtype)) return MOE_ERR_INVALID;
  if ((d_w == nullptr) != (d_recv_w == nullptr)) return MOE_ERR_INVALID;
  if (!aligned(d_w, 4) || !aligned(d_recv_w, 4)) return MOE_ERR_INVALID;
  const int64_t row_bytes = static_cast<int64_t>(H) * elt_bytes(dtype);
  return from_cuda(
      moe::launch_dispatch(h, d_x, row_bytes, d_w, d_recv, d_recv_w, d_send, as_stream(stream)));
}

moe_status moe_combine(const moe_handle* h, const void* d_y, int32_t H, int32_t dtype,
                       const float* d_w, void* d_out, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_y, H, dtype) || !row_ok(d_out, H, dtype) || !aligned(d_w, 4))
    return MOE_ERR_INVALID;
  return from_cuda(moe::launch_combine(h, d_y, H, dtype, d_w, d_out, as_stream(stream)));
}

moe_status moe_combine_bwd(const moe_handle* h, const void* d_g, const void* d_y, int32_t H,
                           int32_t dtype, const float* d_w, void* d_gy, float* d_gw,
                           void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_g, H, dtype) || !row_ok(d_gy, H, dtype)) return MOE_ERR_INVALID;
  if (d_w && d_gw && !row_ok(d_y, H, dtype)) return MOE_ERR_INVALID;
  if (!aligned(d_w, 4) || !aligned(d_gw, 4)) return MOE_ERR_INVALID;
  return from_cuda(
      moe::launch_combine_bwd(h, d_g, d_y, H, dtype, d_w, d_gy, d_gw, as_stream(stream)));
}

moe_status moe_dispatch_bwd(const moe_handle* h, const void* d_grecv, int32_t H, int32_t dtype,
                            void* d_gx, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_grecv, H, dtype) || !row_ok(d_gx, H, dtype)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_combine(h, d_grecv, H, dtype, nullptr, d_gx, as_stream(stream)));
}

moe_status moe_dispatch_bwd_route(const moe_handle* h, const void* d_grecv, int32_t H,
                                  int32_t dtype, const float* d_logits, const int32_t* d_idx,
                                  const float* d_gw, void* d_gx, float* d_glogits, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_grecv, H, dtype) || !row_ok(d_gx, H, dtype)) return MOE_ERR_INVALID;
  if (!d_logits || !d_idx || !d_gw || !d_glogits) return MOE_ERR_INVALID;
  if (!aligned(d_logits, 4) || !aligned(d_idx, 4) || !aligned(d_gw, 4) || !aligned(d_glogits, 4))
    return MOE_ERR_INVALID;
  return from_cuda(moe::launch_dispatch_bwd_route(h, d_grecv, H, dtype, d_logits, d_idx, d_gw,
                                                  d_gx, d_glogits, as_stream(stream)));
}

moe_status moe_dispatch_bwd_route_launches(const moe_handle* h, int32_t* n_launches) {
  if (!h || !n_launches) return MOE_ERR_INVALID;
  *n_launches = moe::dispatch_bwd_route_launches(h->cfg);
  return MOE_OK;
}

moe_status moe_expand(const moe_handle* h, const void* d_send, int32_t H, int32_t dtype,
                      void* d_recv, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_send, H, dtype) || !row_ok(d_recv, H, dtype)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_staged(0, h, d_send, H, dtype, nullptr, d_recv, as_stream(stream)));
}

moe_status moe_combine_partial(const moe_handle* h, const void* d_y, int32_t H, int32_t dtype,
                               const float* d_w, void* d_partial, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_y, H, dtype) || !row_ok(d_partial, H, dtype) || !aligned(d_w, 4))
    return MOE_ERR_INVALID;
  return from_cuda(moe::launch_staged(1, h, d_y, H, dtype, d_w, d_partial, as_stream(stream)));
}

moe_status moe_combine_reduce(const moe_handle* h, const void* d_partial, int32_t H,
                              int32_t dtype, void* d_out, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(H, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_partial, H, dtype) || !row_ok(d_out, H, dtype)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_staged(2, h, d_partial, H, dtype, nullptr, d_out, as_stream(stream)));
}

moe_status moe_scale_rows(const moe_handle* h, const void* d_h, int32_t I, int32_t dtype,
                          const float* d_recv_w, void* d_hs, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(I, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_h, I, dtype) || !row_ok(d_hs, I, dtype)) return MOE_ERR_INVALID;
  if (!d_recv_w || !aligned(d_recv_w, 4)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_scale_rows(h, d_h, I, dtype, d_recv_w, d_hs, as_stream(stream)));
}

moe_status moe_scale_rows_bwd(const moe_handle* h, const void* d_ghs, const void* d_h, int32_t I,
                              int32_t dtype, const float* d_recv_w, void* d_gh, float* d_gw,
                              void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (h->T == 0) return empty_rows_ok(I, dtype) ? MOE_OK : MOE_ERR_INVALID;
  if (!row_ok(d_ghs, I, dtype) || !row_ok(d_h, I, dtype) || !row_ok(d_gh, I, dtype))
    return MOE_ERR_INVALID;
  if (!d_recv_w || !aligned(d_recv_w, 4) || !d_gw || !aligned(d_gw, 4)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_scale_rows_bwd(h, d_ghs, d_h, I, dtype, d_recv_w, d_gh, d_gw,
                                              as_stream(stream)));
}

moe_status moe_dispatch_layout_launches(const moe_handle* h, int32_t T, int32_t* n_launches) {
  if (!h || !n_launches || T < 0) return MOE_ERR_INVALID;
  if (T > h->cfg.max_tokens) return MOE_ERR_CAPACITY;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return MOE_ERR_CUDA;
  *n_launches = moe::layout_launches(h->cfg, T);
  if (prev != h->device) cudaSetDevice(prev);
  return MOE_OK;
}

moe_status moe_w2_absorbed(const moe_handle* h, const void* d_h, int32_t I, const float* d_recv_w,
                           const void* d_w2, int32_t H, void* d_y, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  if (!moe::w2_shape_ok(I, H)) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(h->cfg.num_experts) * H > INT32_MAX) return MOE_ERR_INVALID;
  if (h->T < 0) return MOE_ERR_STATE;
  if (static_cast<int64_t>(h->T) * h->cfg.top_k + static_cast<int64_t>(h->cfg.num_experts) * (h->pad - 1) == 0)
    return MOE_OK;
  if (!d_h || !d_w2 || !d_y) return MOE_ERR_INVALID;
  if (!aligned(d_h, 16) || !aligned(d_w2, 16) || !aligned(d_y, 16)) return MOE_ERR_INVALID;
  if (!d_recv_w || !aligned(d_recv_w, 4)) return MOE_ERR_INVALID;
  return from_cuda(moe::launch_w2_absorbed(h, d_h, I, d_recv_w, d_w2, H, d_y, as_stream(stream)));
}

moe_status moe_read_device_status(const moe_handle* h, uint32_t* host_flags) {
  if (!h || !host_flags) return MOE_ERR_INVALID;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_flags, h->flags, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (prev != h->device) cudaSetDevice(prev);
  return from_cuda(e);
}

moe_status moe_clear_device_status(moe_handle* h, void* stream) {
  if (!h) return MOE_ERR_INVALID;
  if (!on_handle_device(h)) return MOE_ERR_INVALID;
  cudaError_t e = cudaMemsetAsync(h->flags, 0, sizeof(uint32_t), as_stream(stream));
  // a layout whose hand-over timed out left its arrival counter short of
  // zero-on-exit: re-arm it (the epoch word is only ever compared relatively)
  if (e == cudaSuccess) e = cudaMemsetAsync(h->ticket, 0, sizeof(uint32_t), as_stream(stream));
  return from_cuda(e);
}

moe_status moe_set_wait_limit(moe_handle* h, uint64_t limit_ns) {
  if (!h) return MOE_ERR_INVALID;
  h->wait_ns = limit_ns ? limit_ns : MOE_DEFAULT_WAIT_LIMIT_NS;
  return MOE_OK;
}

}  // extern "C"
