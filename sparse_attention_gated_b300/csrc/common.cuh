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

// Absolute position of query j of row `row` (row = b * n_q + j): the caller's per-query
// position where an array of them is given (device memory), else q_pos0 + j.
__device__ __forceinline__ int64_t query_pos(const int64_t* q_pos, int64_t q_pos0, int64_t row, int64_t j) {
  return q_pos != nullptr ? __ldg(q_pos + row) : q_pos0 + j;
}

// Entries visible to position t, at most the n_entries that exist.  The host checks
// every position it is given as a number; a position read from device memory that is
// negative or would see more entries than exist is reported as HYB_DEV_BAD_INDEX and
// clipped (a negative one sees nothing).
__device__ __forceinline__ int64_t visible_checked(int64_t t, int64_t m, int64_t n_entries, int32_t* dev_status,
                                                   bool report) {
  if (t < 0) {
    if (report) flag_status(dev_status, HYB_DEV_BAD_INDEX);
    return 0;
  }
  const int64_t v = visible_entries(t, m);
  if (v > n_entries) {
    if (report) flag_status(dev_status, HYB_DEV_BAD_INDEX);
    return n_entries;
  }
  return v;
}

// The sliding window of position t: absolute rows max(0, t-n_win+1) .. t of a buffer
// whose row 0 is absolute position kv_pos0 and which holds n_kv rows.  Returns the row
// count and sets *first to the buffer row of the first one.  Rows outside the buffer
// (possible only with positions read from device memory: the host checks its own) are
// left out and reported as HYB_DEV_BAD_INDEX.
__device__ __forceinline__ int64_t window_rows(int64_t t, int64_t n_win, int64_t kv_pos0, int64_t n_kv,
                                               int64_t* first, int32_t* dev_status, bool report) {
  int64_t lo = t - n_win + 1 > 0 ? t - n_win + 1 : 0;
  int64_t hi = t;
  bool bad = t < 0;
  if (lo < kv_pos0) lo = kv_pos0, bad = true;
  if (hi > kv_pos0 + n_kv - 1) hi = kv_pos0 + n_kv - 1, bad = true;
  if (bad && report) flag_status(dev_status, HYB_DEV_BAD_INDEX);
  if (hi < lo) {
    *first = 0;
    return 0;
  }
  *first = lo - kv_pos0;
  return hi - lo + 1;
}

}  // namespace hyb
