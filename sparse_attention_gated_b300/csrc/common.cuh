// common.cuh -- small device helpers shared by the hybrid-attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hyb.h"

namespace hyb {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kNumSMs = 148;  // B300: two dies x 74 SMs

__device__ __forceinline__ float exp2_approx(float x) { return exp2f(x); }

// ------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream serialization
// (launch_pdl), so it may be scheduled while the kernel before it in the stream is
// still finishing.  Each kernel calls pdl_wait() before its first access to global
// memory (from then on it sees every write of the kernels before it, whoever
// launched them) and pdl_trigger() once its successor may be scheduled; setup that
// touches only shared memory, TMEM and kernel parameters runs before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------- vector loads
// load_vec<V>(p, x): V consecutive elements starting at p (aligned to their
// total size, or 16 bytes if smaller) converted to float.

template <int V>
__device__ __forceinline__ void load_vec(const float* __restrict__ p, float (&x)[V]) {
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4) {
      float4 t = __ldg(reinterpret_cast<const float4*>(p + i));
      x[i] = t.x, x[i + 1] = t.y, x[i + 2] = t.z, x[i + 3] = t.w;
    }
  } else if constexpr (V % 2 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 2) {
      float2 t = __ldg(reinterpret_cast<const float2*>(p + i));
      x[i] = t.x, x[i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) x[i] = __ldg(p + i);
  }
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t u, float& a, float& b) {
  a = __uint_as_float(u << 16);
  b = __uint_as_float(u & 0xFFFF0000u);
}

template <int V>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* __restrict__ p, float (&x)[V]) {
  if constexpr (V % 8 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 8) {
      uint4 t = __ldg(reinterpret_cast<const uint4*>(p + i));
      bf16x2_to_f32(t.x, x[i], x[i + 1]);
      bf16x2_to_f32(t.y, x[i + 2], x[i + 3]);
      bf16x2_to_f32(t.z, x[i + 4], x[i + 5]);
      bf16x2_to_f32(t.w, x[i + 6], x[i + 7]);
    }
  } else if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4) {
      uint2 t = __ldg(reinterpret_cast<const uint2*>(p + i));
      bf16x2_to_f32(t.x, x[i], x[i + 1]);
      bf16x2_to_f32(t.y, x[i + 2], x[i + 3]);
    }
  } else if constexpr (V % 2 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 2) {
      uint32_t t = __ldg(reinterpret_cast<const unsigned int*>(p + i));
      bf16x2_to_f32(t, x[i], x[i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) x[i] = __bfloat162float(p[i]);
  }
}

// ---------------------------------------------------------------- stores
template <int V>
__device__ __forceinline__ void store_vec(float* p, const float (&x)[V]) {
  if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
  } else if constexpr (V % 2 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 2) *reinterpret_cast<float2*>(p + i) = make_float2(x[i], x[i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) p[i] = x[i];
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int V>
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&x)[V]) {
  if constexpr (V % 8 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 8)
      *reinterpret_cast<uint4*>(p + i) = make_uint4(pack_bf16x2(x[i], x[i + 1]), pack_bf16x2(x[i + 2], x[i + 3]),
                                                    pack_bf16x2(x[i + 4], x[i + 5]), pack_bf16x2(x[i + 6], x[i + 7]));
  } else if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4)
      *reinterpret_cast<uint2*>(p + i) = make_uint2(pack_bf16x2(x[i], x[i + 1]), pack_bf16x2(x[i + 2], x[i + 3]));
  } else if constexpr (V % 2 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 2) *reinterpret_cast<uint32_t*>(p + i) = pack_bf16x2(x[i], x[i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) p[i] = __float2bfloat16_rn(x[i]);
  }
}

// ---------------------------------------------------------------- reductions
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

// Order-preserving map of a float32 onto uint32 (larger float -> larger key).
// -0 is folded onto +0 first so that equal values get equal keys.
__device__ __forceinline__ uint32_t float_order_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void flag_status(int32_t* dev_status, int bits) {
  if (dev_status) atomicOr(reinterpret_cast<int*>(dev_status), bits);
}

// Entries visible to absolute position t with compression factor m.
__host__ __device__ __forceinline__ int64_t visible_entries(int64_t t, int64_t m) { return (t + 1) / m; }

}  // namespace hyb
