// Shared device helpers of the MoE routing library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"

namespace moe {

// ---------------------------------------------------------------------------
// status word

__device__ __forceinline__ void raise_flag(uint32_t* flags, uint32_t bit) {
  if (flags) atomicOr(flags, bit);
}

// A row index read from the layout (a receive row, a send row), checked
// against the n rows of the tensor it indexes: -1 (a dropped entry) stays -1;
// any other index outside [0, n) raises MOE_DEVERR_BAD_LAYOUT and reads as -1,
// so that the entry is skipped instead of reaching outside the tensor.
__device__ __forceinline__ int checked_row(int r, int n, uint32_t* flags) {
  if (static_cast<unsigned>(r) < static_cast<unsigned>(n)) return r;
  if (r != -1) raise_flag(flags, MOE_DEVERR_BAD_LAYOUT);
  return -1;
}

// ---------------------------------------------------------------------------
// 16-byte vector rows

struct alignas(16) Vec16 {
  uint32_t u[4];
};

// Streaming 16-byte load of data read once: non-coherent path, no L1
// allocation.
__device__ __forceinline__ Vec16 ld_stream(const void* p) {
  Vec16 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3])
               : "l"(p));
  return v;
}

// 16-byte load through L1 (coherent path, default caching).  The combine
// backward's gathered expert-output rows, the dispatch's token rows and the
// absorption backward's gathered rows load faster this way than by the
// non-coherent path without L1 allocation (DeepSeek-V3 shape: combine
// backward 616.6 against 630.1 us a launch; Qwen3-235B shape: the step 2140
// against 2149 us).
__device__ __forceinline__ Vec16 ld_vec(const void* p) {
  Vec16 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.u[0]), "=r"(v.u[1]), "=r"(v.u[2]), "=r"(v.u[3])
               : "l"(p));
  return v;
}

// 16-byte store with the evict-first (streaming) policy: the dispatch's K
// receive rows of each token (315.8 against 317.9 us a launch).
__device__ __forceinline__ void st_vec_cs(void* p, const Vec16& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.u[0]), "r"(v.u[1]),
               "r"(v.u[2]), "r"(v.u[3])
               : "memory");
}

__device__ __forceinline__ void st_vec(void* p, const Vec16& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.u[0]), "r"(v.u[1]),
               "r"(v.u[2]), "r"(v.u[3])
               : "memory");
}

// Element access of a 16-byte vector as fp32 (bf16: 8 elements, f32: 4).
template <typename Elt>
struct VecTraits;

template <>
struct VecTraits<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void to_f32(const Vec16& v, float* f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(v.u[i] << 16);
      f[2 * i + 1] = __uint_as_float(v.u[i] & 0xffff0000u);
    }
  }
  // round-to-nearest-even of each fp32 value
  __device__ __forceinline__ static Vec16 from_f32(const float* f) {
    Vec16 v;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      v.u[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    return v;
  }
};

template <>
struct VecTraits<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void to_f32(const Vec16& v, float* f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(v.u[i]);
  }
  __device__ __forceinline__ static Vec16 from_f32(const float* f) {
    Vec16 v;
#pragma unroll
    for (int i = 0; i < 4; ++i) v.u[i] = __float_as_uint(f[i]);
    return v;
  }
};

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: the routing, layout and dispatch kernels are
// launched (by launch_chained) so that a kernel's blocks may be scheduled
// while the previous grid drains, which hides most of the launch gap after
// the short routing and layout kernels; each such kernel first lets its own
// successor do the same, then waits until the previous grid has completed
// and its memory is visible, before any global access.

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.launch_dependents;\n\tgriddepcontrol.wait;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization (and, with
// `cooperative`, as a cooperative grid).  The kernel must begin with
// grid_dependency_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t s, bool cooperative, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = cooperative ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// warp helpers

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe
