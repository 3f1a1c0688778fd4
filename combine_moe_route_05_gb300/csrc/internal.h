// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"


struct moe_handle {
  moe_config cfg;
  int device;
  int num_sms;
  long long l2_bytes;  // the device's L2 cache
  int T;  // tokens of the current layout, -1 before the first
  int max_tiles;
  int pad;  // receive segments rounded up to a multiple of pad rows (>= 1)
  unsigned long long wait_ns;  // limit of the kernels' bounded waits
  uint32_t* flags;   // device status word (MOE_DEVERR_* bits)
  uint32_t* ticket;  // the layout's tile hand-over: [0] arrivals, [1] epoch (one 64-bit word)
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
  int32_t* tile_hist;  // [(E + R) columns][max_tiles], exclusive tile bases after the scan
};

namespace moe {

// Resident blocks per SM of `kernel` at `threads` threads and `smem` dynamic
// shared memory (cached per kernel).
int resident_blocks(const void* kernel, int threads, size_t smem);

cudaError_t launch_route_topk(const moe_handle* h, const float* logits, const float* bias, int T,
                              int32_t* idx, float* w, cudaStream_t s);

cudaError_t launch_route_bwd(const moe_handle* h, const float* logits, const int32_t* idx,
                             const float* gw, int T, float* glogits, cudaStream_t s);

cudaError_t launch_layout(const moe_handle* h, const int32_t* idx, int T, cudaStream_t s);

cudaError_t launch_dispatch(const moe_handle* h, const void* x, int64_t row_bytes, const float* w,
                            void* recv, float* recv_w, void* send, cudaStream_t s);

cudaError_t launch_combine(const moe_handle* h, const void* y, int H, int dtype, const float* w,
                           void* out, cudaStream_t s);

cudaError_t launch_combine_bwd(const moe_handle* h, const void* g, const void* y, int H, int dtype,
                               const float* w, void* gy, float* gw, cudaStream_t s);

// Router inputs and output of the dispatch backward with the router backward
// to the logits fused in (softmax with renormalisation or sigmoid).
struct RouterBwdRows {
  const float* logits;  // [T, E]
  const int32_t* idx;   // [T, K]
  const float* gw;      // [T, K], complete
  float* glogits;       // [T, E]
};

// dispatch backward (unit-weight combine of grecv into gx) and router
// backward in one launch when the configuration allows it (every routing but
// softmax without renormalisation), else the two kernels back to back
cudaError_t launch_dispatch_bwd_route(const moe_handle* h, const void* grecv, int H, int dtype,
                                      const float* logits, const int32_t* idx, const float* gw,
                                      void* gx, float* glogits, cudaStream_t s);

// launches launch_dispatch_bwd_route makes (1 or 2) for the handle's routing
int dispatch_bwd_route_launches(const moe_config& c);

// op 0: expand send rows to receive rows; 1: combine into per-send-row
// partials; 2: reduce the partials to token rows
cudaError_t launch_staged(int op, const moe_handle* h, const void* src, int H, int dtype,
                          const float* w, void* dst, cudaStream_t s);

// Writes zeros to the pad rows of a receive-row tensor (rows of row_bytes,
// a multiple of 4) when the layout is padded; nothing otherwise.
cudaError_t zero_pad_rows(const moe_handle* h, void* rows, int64_t row_bytes, cudaStream_t s);

cudaError_t launch_scale_rows(const moe_handle* h, const void* hrows, int I, int dtype,
                              const float* recv_w, void* hs, cudaStream_t s);

cudaError_t launch_scale_rows_bwd(const moe_handle* h, const void* ghs, const void* hrows, int I,
                                  int dtype, const float* recv_w, void* gh, float* gw,
                                  cudaStream_t s);

int layout_launches(const moe_config& c, int T);
cudaError_t prepare_w2_kernel();
bool w2_shape_ok(int I, int H);
// Bounded waits inside the kernels give up after this long by default (1 s).
#define MOE_DEFAULT_WAIT_LIMIT_NS 1000000000ull

cudaError_t launch_w2_absorbed(const moe_handle* h, const void* hrows, int I, const float* recv_w,
                               const void* w2, int H, void* y, cudaStream_t s);

}  // namespace moe
