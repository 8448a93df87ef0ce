// Shared device/host helpers for the MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/moe.h"

namespace moe {

// One-time per-device set-up on the host (function attributes, occupancy queries,
// symbol addresses), safe for callers on several host threads.  The first caller on
// a device runs init() under one library-wide lock; the flag is then published with
// release order and read with acquire order, so a caller that finds it set also sees
// everything init() wrote.  A failed init() leaves the flag clear (the next call
// retries).  Devices at or above N are not cached: init() runs on every call.
inline std::mutex& setup_mutex() {
  static std::mutex m;
  return m;
}
template <int N>
struct OncePerDevice {
  std::atomic<bool> done[N] = {};
  template <class F>
  cudaError_t run(int dev, F&& init) {
    if (dev < 0 || dev >= N) return init();
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(setup_mutex());
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = init();
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
  }
};

// Status codes recorded on the device (a per-device word; see moe_api.cu).
// The first condition wins; later ones are dropped until the host reads it.
__device__ __forceinline__ void record_status(unsigned* status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded waits give up after this long (the kernels' longest legitimate wait
// is well under a millisecond).  The fault-injection test build (MOE_FAULT_INJECTION,
// libmoe_fault.so; never the product library) gives up after 50 ms.
#ifdef MOE_FAULT_INJECTION
constexpr uint64_t kWaitLimitNs = 50000000ull;  // 50 ms
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
#endif

template <typename T> struct Act;
template <> struct Act<float> {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ static float to_f(float v) { return v; }
  __device__ static float from_f(float v) { return v; }
};
template <> struct Act<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector of activations, unpacked to fp32.
template <typename T>
__device__ __forceinline__ void load_vec_f32(const T* p, float* out);
template <>
__device__ __forceinline__ void load_vec_f32<float>(const float* p, float* out) {
  float4 v = *reinterpret_cast<const float4*>(p);
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec_f32<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x; out[2 * i + 1] = f.y;
  }
}

template <typename T>
__device__ __forceinline__ void store_vec_f32(T* p, const float* in);
template <>
__device__ __forceinline__ void store_vec_f32<float>(float* p, const float* in) {
  *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
}
template <>
__device__ __forceinline__ void store_vec_f32<__nv_bfloat16>(__nv_bfloat16* p, const float* in) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = v;
}

// The same with streaming cache hints (data read or written once: evict first).
template <typename T>
__device__ __forceinline__ void load_vec_f32_cs(const T* p, float* out);
template <>
__device__ __forceinline__ void load_vec_f32_cs<float>(const float* p, float* out) {
  const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
template <>
__device__ __forceinline__ void load_vec_f32_cs<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
  uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x; out[2 * i + 1] = f.y;
  }
}
template <typename T>
__device__ __forceinline__ void store_vec_f32_cs(T* p, const float* in);
template <>
__device__ __forceinline__ void store_vec_f32_cs<float>(float* p, const float* in) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(in[0], in[1], in[2], in[3]));
}
template <>
__device__ __forceinline__ void store_vec_f32_cs<__nv_bfloat16>(__nv_bfloat16* p, const float* in) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Kernels of the layer are launched with
// programmatic stream serialization: a kernel may be scheduled while the one
// before it on the stream is finishing.  Each such kernel calls pdl_trigger()
// early (its own dependent may then be scheduled once all of its blocks have
// started) and pdl_wait() before its first global-memory access; pdl_wait
// returns once the preceding grid has completed and its writes are visible.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
