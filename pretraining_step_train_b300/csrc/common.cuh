// Device-side helpers shared by the GPT-2 step kernels (sm_103a).
#pragma once
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

// Bits of the device status word (latched, read back by the host).
#define ST_TOKEN 1u      // a token id outside [0, V) was clamped
#define ST_TIMEOUT 2u    // a bounded wait in a pipelined kernel gave up
#define ST_NONFINITE 4u  // a non-finite loss or gradient norm was seen

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct V16 { static constexpr int N = 16 / sizeof(T); };

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* out) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 4) {
    out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
  } else {
    const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = __bfloat162float(h[i]);
  }
}

template <typename T>
__device__ __forceinline__ void store16(T* p, const float* in) {
  uint4 u;
  if constexpr (sizeof(T) == 4) {
    u.x = __float_as_uint(in[0]); u.y = __float_as_uint(in[1]);
    u.z = __float_as_uint(in[2]); u.w = __float_as_uint(in[3]);
  } else {
    bf16* h = reinterpret_cast<bf16*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __float2bfloat16_rn(in[i]);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// Streaming (evict-first) 16-byte load for data read exactly once.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// tanh-form GELU and its derivative (Hendrycks & Gimpel), evaluated in fp32.
#define GELU_K 0.7978845608028654f
#define GELU_C 0.044715f
__device__ __forceinline__ float gelu_f(float x) {
  float u = GELU_K * (x + GELU_C * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}
__device__ __forceinline__ float gelu_grad_f(float x) {
  float u = GELU_K * (x + GELU_C * x * x * x);
  float th = tanhf(u);
  float du = GELU_K * (1.0f + 3.0f * GELU_C * x * x);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * du;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  Every kernel of this library is launched by
// launch_k with programmatic stream serialization allowed: once all CTAs of
// the previous kernel on the stream have exited, this kernel's CTAs may be
// scheduled before that grid's completion is processed.  Each kernel waits
// until its predecessor has completed and its writes are visible (pdl_wait)
// before it reads or writes global memory or allocates tensor memory.  No
// kernel triggers its successor early (CTAs that wait while a predecessor
// still runs took issue slots from it), so only the launch latency overlaps.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() { pdl_wait(); }

// Launch configuration of launch_k; `pair` adds a cluster dimension of 2 (CTA pairs).
inline cudaLaunchConfig_t launch_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
                                     bool pair) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  return cfg;
}

// As launch_k, in clusters of two CTAs (grid.x even).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_pair(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 Args&&... args) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_cfg(grid, block, smem, s, attr, true);
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
