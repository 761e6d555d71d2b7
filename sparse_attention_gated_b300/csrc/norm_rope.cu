// norm_rope.cu -- RMSNorm of a row, then rotary encoding of its last
// rope_dims dimensions ("DeepSeek-V4 hybrid attention" (trishampatil.com)
// section IV; rotary convention of the PyTorch walkthrough on juhe.plus, "The
// Code: RoPE Helpers": consecutive pairs, frequencies theta^(-2i/d)).
//
// One warp per row, in place.  Pass 1: the sum of squares (each lane a stride
// of pairs, warp reduction).  Pass 2: scale by 1/sqrt(mean + eps) and gamma,
// then rotate the pairs of the last rope_dims dimensions.  The angle
// pos * theta^(-2i/d) can reach 10^6 rad: it is formed in float64 and reduced
// modulo 2 pi there, and only the reduced angle goes to float32 sin / cos.
// Float64 is slow on this part, so the frequency theta^(-2i/d) is the host's
// float64 base theta^(-2/d) raised to the integer i by repeated squaring (at
// most 8 squarings), and the reduction subtracts k = rint(angle / 2 pi) times
// 2 pi split into two float64 parts (Cody and Waite's additive reduction): a
// few float64 operations per rotated pair instead of a general power and a
// remainder.
#include <cmath>

#include "kernels.cuh"

namespace hyb {

struct NormRopeParams {
  void* x;
  int64_t rows, c;
  const float* gamma;
  float eps;
  const int64_t* pos;
  int64_t rows_per_pos, rope_dims;
  double rope_base;    // theta^(-2 / rope_dims)
  int64_t row_stride;  // elements from one row to the next
};

template <typename T>
__device__ __forceinline__ float2 ld_pair(const T* p);
template <>
__device__ __forceinline__ float2 ld_pair<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 ld_pair<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// Row r of a call (one warp).
template <typename T>
__device__ __forceinline__ void norm_rope_row(const NormRopeParams& p, int64_t r, int lane) {
  T* x = static_cast<T*>(p.x) + r * p.row_stride;
  const int64_t n_pairs = p.c / 2;
  float ss = 0.f;
  for (int64_t i = lane; i < n_pairs; i += 32) {
    const float2 v = ld_pair<T>(x + 2 * i);
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, ss));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)p.c + p.eps);
  const int64_t first_rot = (p.c - p.rope_dims) / 2;  // first rotated pair
  const double pos = p.rope_dims > 0 ? (double)p.pos[r / p.rows_per_pos] : 0.0;
  // 2 pi = kTwoPiHi + kTwoPiLo (the float64 nearest 2 pi and the remainder)
  constexpr double kTwoPiHi = 6.283185307179586232, kTwoPiLo = 2.4492935982947064e-16;
  constexpr double kInvTwoPi = 0.15915494309189535;
  for (int64_t i = lane; i < n_pairs; i += 32) {
    float2 v = ld_pair<T>(x + 2 * i);
    const float g0 = p.gamma ? p.gamma[2 * i] : 1.f, g1 = p.gamma ? p.gamma[2 * i + 1] : 1.f;
    v.x = v.x * inv * g0;
    v.y = v.y * inv * g1;
    if (i >= first_rot) {
      double freq = 1.0, b = p.rope_base;
      for (int64_t e = i - first_rot; e > 0; e >>= 1) {  // rope_base^(i - first_rot)
        if (e & 1) freq *= b;
        b *= b;
      }
      const double a = pos * freq;
      const double k = rint(a * kInvTwoPi);
      const float ang = (float)fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, a));
      float sn, cs;
      sincosf(ang, &sn, &cs);
      v = make_float2(v.x * cs - v.y * sn, v.x * sn + v.y * cs);
    }
    st_pair(x + 2 * i, v);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) norm_rope_kernel(NormRopeParams p) {
  pdl_wait();
  pdl_trigger();
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (r >= p.rows) return;
  norm_rope_row<T>(p, r, threadIdx.x & 31);
}

// Several calls of one dtype in one launch: call i takes blocks [block_end[i-1], block_end[i]).
struct NormRopeBatch {
  NormRopeParams call[kNormRopeBatchMax];
  int64_t block_end[kNormRopeBatchMax];
  int n;
};

template <typename T>
__global__ void __launch_bounds__(256) norm_rope_batch_kernel(NormRopeBatch b) {
  pdl_wait();
  pdl_trigger();
  int i = 0;
  while (i + 1 < b.n && (int64_t)blockIdx.x >= b.block_end[i]) ++i;
  const int64_t blk = (int64_t)blockIdx.x - (i > 0 ? b.block_end[i - 1] : 0);
  const NormRopeParams& p = b.call[i];
  const int64_t r = (blk * blockDim.x + threadIdx.x) >> 5;
  if (r >= p.rows) return;
  norm_rope_row<T>(p, r, threadIdx.x & 31);
}

static NormRopeParams norm_rope_params(const hyb_norm_rope_args* a) {
  NormRopeParams p;
  p.x = a->x, p.rows = a->rows, p.c = a->c, p.gamma = a->gamma, p.eps = a->eps, p.pos = a->pos;
  p.rows_per_pos = a->rows_per_pos, p.rope_dims = a->rope_dims;
  p.rope_base = a->rope_dims > 0 ? std::pow(a->theta, -2.0 / (double)a->rope_dims) : 1.0;
  p.row_stride = a->row_stride > 0 ? a->row_stride : a->c;
  return p;
}

cudaError_t launch_norm_rope_batch(const hyb_norm_rope_args* calls, int n, cudaStream_t s) {
  NormRopeBatch b{};
  int64_t blocks = 0;
  b.n = 0;
  for (int i = 0; i < n; ++i) {
    if (calls[i].rows == 0) continue;
    b.call[b.n] = norm_rope_params(&calls[i]);
    blocks += (calls[i].rows + 7) / 8;
    b.block_end[b.n] = blocks;
    ++b.n;
  }
  if (b.n == 0) return cudaSuccess;
  if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e = calls[0].dtype == HYB_F32
                      ? launch_pdl(norm_rope_batch_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, b)
                      : launch_pdl(norm_rope_batch_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, s, b);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_norm_rope(const hyb_norm_rope_args* a, cudaStream_t s) {
  const NormRopeParams p = norm_rope_params(a);
  if (p.rows == 0) return cudaSuccess;
  const int64_t blocks = (p.rows + 7) / 8;
  if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e = a->dtype == HYB_F32 ? launch_pdl(norm_rope_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, p)
                                      : launch_pdl(norm_rope_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256),
                                                   0, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
