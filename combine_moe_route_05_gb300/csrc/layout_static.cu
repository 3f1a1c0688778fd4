// Allocation-free dispatch layout: moe_dispatch_layout_static.
//
// Same kernels as moe_dispatch_layout, but the scratch they need (the arrival
// ticket of the last-block scan and the per-tile counters) lives in a
// file-scope device array instead of a caller-allocated workspace, and the
// outputs go to caller-owned arrays.  For callers that may not allocate
// device memory at all -- for example a plugin whose host framework hands it
// only its input and output buffers and forbids cudaMalloc on the execution
// path (a cudaMalloc there synchronises the device and is not allowed while
// the framework captures the stream).
#include <mutex>

#include "internal.h"

namespace moe {
bool valid_config(const moe_config* c);
cudaError_t prepare_layout_kernels();
int layout_tiles(int T);
cudaError_t launch_layout_buffers(const moe_config& c, const int32_t* idx, int T,
                                  const moe_layout& out, uint32_t* flags, uint32_t* ticket,
                                  int32_t* tile_hist, int max_tiles, unsigned long long wait_ns,
                                  cudaStream_t s);
}  // namespace moe

namespace {

constexpr int kTicketSlot = 64;  // int32 words before the counters (keeps them 256-byte aligned)
constexpr int kCapacity = MOE_LAYOUT_STATIC_COUNTERS;
constexpr int kMaxDevices = 64;

// [0]: arrival ticket; [kTicketSlot, kTicketSlot + kCapacity): tile counters.
// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) int32_t g_layout_scratch[kTicketSlot + kCapacity];

std::mutex g_setup_mu;
int32_t* g_scratch_addr[kMaxDevices];  // device address of g_layout_scratch, per device

// Once per device, with that device current: the device address of the
// scratch array (its host-side name is only a stand-in) and the kernels'
// shared-memory limits.
cudaError_t scratch_of_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    e = moe::prepare_layout_kernels();
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" moe_status moe_dispatch_layout_static(const moe_config* c, const int32_t* d_idx,
                                                 int32_t T, const moe_layout* out,
                                                 uint32_t* d_status, void* stream) {
  if (!moe::valid_config(c) || !out || T < 0) return MOE_ERR_INVALID;
  if (static_cast<int64_t>(T) * c->top_k > INT32_MAX) return MOE_ERR_CAPACITY;
  const int64_t counters =
      static_cast<int64_t>(moe::layout_tiles(T)) * (c->num_experts + c->num_ranks);
  if (counters > kCapacity) return MOE_ERR_CAPACITY;
  const void* always[] = {out->cnt_e, out->off_e, out->cnt_send_r, out->off_send_r,
                          out->cnt_recv_r, out->off_recv_r, out->S};
  for (const void* p : always)
    if (!p || !aligned4(p)) return MOE_ERR_INVALID;
  if (T > 0) {
    const void* rows[] = {d_idx, out->pos, out->recv_token, out->recv_k, out->send_token,
                          out->send_row_of, out->recv_send_row};
    for (const void* p : rows)
      if (!p || !aligned4(p)) return MOE_ERR_INVALID;
  }
  if (!aligned4(d_status)) return MOE_ERR_INVALID;

  int32_t* scratch = nullptr;
  if (scratch_of_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the ticket must start at zero; the counters are fully written before use
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  const int tiles = moe::layout_tiles(T);
  cudaError_t e = moe::launch_layout_buffers(*c, d_idx, T, *out, d_status,
                                             reinterpret_cast<uint32_t*>(scratch),
                                             scratch + kTicketSlot, tiles,
                                             MOE_DEFAULT_WAIT_LIMIT_NS, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
