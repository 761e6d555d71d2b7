// indexer.cu -- lightning-indexer scores on CUDA cores ("DeepSeek-V4 hybrid
// attention" (trishampatil.com) section V.2):
//   I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . K_I[s]),  s < floor((t+1)/m).
//
// One thread per entry s; the block holds query (b, j)'s decoded indexer
// heads (times their scales) and weights in shared memory and every thread
// streams its entry's key row.  Used for the float32 configuration and as the
// general path; the FP8 decode/prefill shapes use the tensor-core kernel.
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace hyb {

struct IndexParams {
  const void* qI;
  const float* qI_scale;
  const float* w;
  const void* kI;
  const float* kI_scale;
  float* scores;
  int64_t score_stride, n_q, n_entries, kv_stride, n_ih, c_I, m, q_pos0;
  const int64_t* q_pos;  // optional per-query positions [batch * n_q]
  int32_t* dev_status;
};

__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& a, float& b) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  a = f.x, b = f.y;
}

template <bool FP8>
__device__ __forceinline__ void load_key16(const void* base, int64_t off, float (&kv)[16]) {
  if constexpr (FP8) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(base) + off));
    uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e4m3x2_to_f32(w4[i], kv[4 * i], kv[4 * i + 1]);
      e4m3x2_to_f32(w4[i] >> 16, kv[4 * i + 2], kv[4 * i + 3]);
    }
  } else {
    load_vec<16>(static_cast<const float*>(base) + off, kv);
  }
}

template <bool FP8, int HG>
__global__ void __launch_bounds__(256) index_scores_cc_kernel(IndexParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float4 smem4[];
  float* q_s = reinterpret_cast<float*>(smem4);  // [n_ih][c_I]
  float* w_s = q_s + p.n_ih * p.c_I;            // [n_ih]
  const int64_t b = blockIdx.z, j = blockIdx.y;
  const int64_t t = query_pos(p.q_pos, p.q_pos0, b * p.n_q + j, j);
  const int64_t vis = visible_checked(t, p.m, p.n_entries, p.dev_status, blockIdx.x == 0 && threadIdx.x == 0);
  const int64_t s0 = (int64_t)blockIdx.x * blockDim.x;
  if (s0 >= vis) return;

  const int64_t qrow = (b * p.n_q + j) * p.n_ih;
  for (int64_t i = threadIdx.x; i < p.n_ih * p.c_I; i += blockDim.x) {
    const int64_t h = i / p.c_I;
    float v;
    if constexpr (FP8) {
      __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<const uint8_t*>(p.qI)[qrow * p.c_I + i], __NV_E4M3);
      v = __half2float(*reinterpret_cast<__half*>(&hr)) * p.qI_scale[qrow + h];
    } else {
      v = static_cast<const float*>(p.qI)[qrow * p.c_I + i];
    }
    q_s[i] = v;
  }
  for (int64_t h = threadIdx.x; h < p.n_ih; h += blockDim.x) w_s[h] = p.w[qrow + h];
  __syncthreads();

  const int64_t s = s0 + threadIdx.x;
  if (s >= vis) return;
  const int64_t krow = (b * p.kv_stride + s) * p.c_I;
  const float ks = FP8 ? p.kI_scale[b * p.kv_stride + s] : 1.0f;
  float score = 0.f;
  for (int64_t hg = 0; hg < p.n_ih; hg += HG) {
    float acc[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) acc[h] = 0.f;
    for (int64_t d0 = 0; d0 < p.c_I; d0 += 16) {
      float kv[16];
      load_key16<FP8>(p.kI, krow + d0, kv);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float4* qq = reinterpret_cast<const float4*>(q_s + (hg + h) * p.c_I + d0);
#pragma unroll
        for (int d4 = 0; d4 < 4; ++d4) {
          float4 qv = qq[d4];
          acc[h] = fmaf(qv.x, kv[4 * d4], acc[h]);
          acc[h] = fmaf(qv.y, kv[4 * d4 + 1], acc[h]);
          acc[h] = fmaf(qv.z, kv[4 * d4 + 2], acc[h]);
          acc[h] = fmaf(qv.w, kv[4 * d4 + 3], acc[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < HG; ++h) score = fmaf(w_s[hg + h], fmaxf(acc[h] * ks, 0.f), score);
  }
  p.scores[(b * p.n_q + j) * p.score_stride + s] = score;
}

bool index_cc_shape_supported(int64_t n_ih, int64_t c_I) {
  return n_ih >= 1 && n_ih <= 256 && (n_ih % 4 == 0) && c_I >= 16 && c_I <= 512 && c_I % 16 == 0;
}

cudaError_t launch_index_scores_cc(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                   cudaStream_t s) {
  IndexParams p;
  p.qI = a->qI, p.qI_scale = a->qI_scale, p.w = a->w, p.kI = a->kI, p.kI_scale = a->kI_scale, p.scores = scores;
  p.score_stride = score_stride, p.n_q = a->n_q, p.n_entries = a->n_entries;
  p.kv_stride = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  p.n_ih = a->n_ih, p.c_I = a->c_I, p.m = a->m, p.q_pos0 = a->q_pos0;
  p.q_pos = a->q_pos, p.dev_status = a->dev_status;
  if (n_vis_max == 0 || a->n_q == 0 || a->batch == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n_vis_max + 255) / 256), (unsigned)a->n_q, (unsigned)a->batch), block(256);
  const size_t smem = sizeof(float) * (size_t)(a->n_ih * a->c_I + a->n_ih) + 16;
  const bool fp8 = a->dtype == HYB_E4M3;
  const bool hg16 = (a->n_ih % 16) == 0;
  auto run = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(kernel, grid, block, smem, s, p);
  };
  cudaError_t e;
  if (fp8 && hg16)
    e = run(index_scores_cc_kernel<true, 16>);
  else if (fp8)
    e = run(index_scores_cc_kernel<true, 4>);
  else if (hg16)
    e = run(index_scores_cc_kernel<false, 16>);
  else
    e = run(index_scores_cc_kernel<false, 4>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
