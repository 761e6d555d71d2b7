// compress.cu -- softmax-gated compressor ("DeepSeek-V4 hybrid attention"
// (trishampatil.com) section V.1 for CSA with overlap, section VI for HCA).
//
// One CTA per (batch, output entry).  The entry's window has W rows (2m with
// overlap, m without).  Threads form a grid of G channel groups (8 channels
// each, one 16-byte bf16 / 32-byte f32 load per row) by R row groups; row
// group g takes window rows g, g+R, g+2R, ...  Each thread keeps, per channel,
// an online softmax (running max, denominator, weighted numerator) in float32
// and base 2 over its rows; the R partial states are then merged in shared
// memory.  Splitting the rows over threads keeps the long HCA window (m' = 128
// rows) from becoming a serial chain of dependent loads.  The kernel is
// HBM-bound: every input row is read once per entry that uses it (CSA rows
// feed two neighbouring entries, stream a of entry i and stream b of entry
// i+1) and each entry is written once.
#include "kernels.cuh"

namespace hyb {

struct CompressParams {
  const void* ca;
  const void* cb;
  const void* za;
  const void* zb;
  const float* bias;
  void* out;
  float* out_scale;
  int64_t batch, n_rows, c, m, first_block, out_batch_stride, n_out, skip;
  int overlap;
  int R;  // row groups
};

constexpr int kCg = 8;  // channels per thread

template <typename Tin>
__device__ __forceinline__ void load8(const Tin* p, float (&x)[kCg]) {
  load_vec<kCg>(p, x);
}

// OUT: 0 = float32, 1 = bf16, 2 = e4m3 + per-entry scale
template <typename Tin, int OUT>
__global__ void __launch_bounds__(512) compress_kernel(CompressParams p) {
  extern __shared__ float sm[];  // [3][R][c]: max, denominator, numerator of each row group
  __shared__ float s_red[32];
  const int64_t c = p.c, m = p.m;
  const int G = (int)(c / kCg);
  const int g = threadIdx.x % G;  // channel group
  const int rg = threadIdx.x / G; // row group
  const int64_t b = blockIdx.x / p.n_out, j = blockIdx.x % p.n_out;
  const int64_t lb = j + p.skip;  // block index within the rows passed in
  const int64_t abs_blk = p.first_block + lb;
  const int64_t ch0 = (int64_t)g * kCg;
  const bool has_prev = p.overlap && abs_blk > 0;
  const int W = (int)(p.overlap ? 2 * m : m);
  const int64_t base = b * p.n_rows;

  float mx[kCg], den[kCg], num[kCg];
#pragma unroll
  for (int i = 0; i < kCg; ++i) mx[i] = -INFINITY, den[i] = 0.f, num[i] = 0.f;

  const Tin* ca = static_cast<const Tin*>(p.ca);
  const Tin* za = static_cast<const Tin*>(p.za);
  const Tin* cb = static_cast<const Tin*>(p.cb);
  const Tin* zb = static_cast<const Tin*>(p.zb);
#pragma unroll 4
  for (int pos = rg; pos < W; pos += p.R) {
    const Tin* zr;
    const Tin* cr;
    if (p.overlap && pos < m) {
      if (!has_prev) continue;  // block -1 does not exist: its logits are -inf
      const int64_t row = base + (lb - 1) * m + pos;
      zr = zb + row * c + ch0, cr = cb + row * c + ch0;
    } else {
      const int64_t row = base + lb * m + (p.overlap ? pos - m : pos);
      zr = za + row * c + ch0, cr = ca + row * c + ch0;
    }
    float z[kCg], cv[kCg], bv[kCg];
    load8<Tin>(zr, z);
    load8<Tin>(cr, cv);
    load_vec<kCg>(p.bias + pos * c + ch0, bv);
#pragma unroll
    for (int i = 0; i < kCg; ++i) {
      const float l = (z[i] + bv[i]) * kLog2e;
      if (l > mx[i]) {
        const float r = exp2f(mx[i] - l);  // 0 when mx = -inf
        den[i] = den[i] * r + 1.0f;
        num[i] = num[i] * r + cv[i];
        mx[i] = l;
      } else {
        const float e = exp2f(l - mx[i]);
        den[i] += e;
        num[i] = fmaf(e, cv[i], num[i]);
      }
    }
  }

  float r[kCg];
  if (p.R > 1) {
    float* s_mx = sm;
    float* s_den = sm + (int64_t)p.R * c;
    float* s_num = s_den + (int64_t)p.R * c;
    const int64_t o = (int64_t)rg * c + ch0;
#pragma unroll
    for (int i = 0; i < kCg; ++i) s_mx[o + i] = mx[i], s_den[o + i] = den[i], s_num[o + i] = num[i];
    __syncthreads();
    if (rg != 0) return;
#pragma unroll
    for (int i = 0; i < kCg; ++i) {
      float M = -INFINITY;
      for (int q = 0; q < p.R; ++q) M = fmaxf(M, s_mx[(int64_t)q * c + ch0 + i]);
      float D = 0.f, N = 0.f;
      for (int q = 0; q < p.R; ++q) {
        const float mq = s_mx[(int64_t)q * c + ch0 + i];
        if (mq == -INFINITY) continue;
        const float f = exp2f(mq - M);
        D = fmaf(f, s_den[(int64_t)q * c + ch0 + i], D);
        N = fmaf(f, s_num[(int64_t)q * c + ch0 + i], N);
      }
      r[i] = N / D;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kCg; ++i) r[i] = num[i] / den[i];
  }

  // only row group 0 (threads 0..G-1) is left here
  const int64_t orow = b * p.out_batch_stride + j;
  if constexpr (OUT == 0) {
    store_vec<kCg>(static_cast<float*>(p.out) + orow * c + ch0, r);
  } else if constexpr (OUT == 1) {
    store_vec<kCg>(static_cast<__nv_bfloat16*>(p.out) + orow * c + ch0, r);
  } else {
    // per-entry scale = amax / 448 over the entry's channels (G threads, G <= 64)
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kCg; ++i) amax = fmaxf(amax, fabsf(r[i]));
    if (G <= 32) {
      // the G threads are lanes 0..G-1 of warp 0 (G is a power of two)
      const unsigned mask = G == 32 ? 0xffffffffu : ((1u << G) - 1u);
      for (int o = G / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(mask, amax, o));
    } else {
      // G = 64: two full warps meet on a named barrier
      amax = warp_max(amax);
      if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
      asm volatile("bar.sync 1, %0;" ::"r"(G) : "memory");
      amax = 0.f;
      for (int w = 0; w < G / 32; ++w) amax = fmaxf(amax, s_red[w]);
    }
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < kCg; ++i) {
      const uint32_t code = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(r[i], scale), __NV_SATFINITE, __NV_E4M3);
      if (i < 4)
        lo |= code << (8 * i);
      else
        hi |= code << (8 * (i - 4));
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + orow * c + ch0) = make_uint2(lo, hi);
    if (threadIdx.x == 0) p.out_scale[orow] = scale;
  }
}

template <typename Tin>
static cudaError_t launch_t(CompressParams& p, int out_dtype, cudaStream_t s) {
  const int G = (int)(p.c / kCg);
  const int W = (int)(p.overlap ? 2 * p.m : p.m);
  int R = 512 / G;
  if (R > W) R = W;
  if (R < 1) R = 1;
  p.R = R;
  const size_t smem = R > 1 ? (size_t)3 * R * p.c * sizeof(float) : 0;
  const dim3 grid((unsigned)(p.batch * p.n_out)), block((unsigned)(G * R));
  cudaError_t e = cudaSuccess;
  if (out_dtype == HYB_F32) {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) compress_kernel<Tin, 0><<<grid, block, smem, s>>>(p);
  } else if (out_dtype == HYB_BF16) {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) compress_kernel<Tin, 1><<<grid, block, smem, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) compress_kernel<Tin, 2><<<grid, block, smem, s>>>(p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool compress_shape_supported(int64_t c) { return c == 32 || c == 64 || c == 128 || c == 256 || c == 512; }

cudaError_t launch_compress(const hyb_compress_args* a, int64_t n_out, cudaStream_t s) {
  CompressParams p;
  p.ca = a->ca, p.cb = a->cb, p.za = a->za, p.zb = a->zb, p.bias = a->bias, p.out = a->out, p.out_scale = a->out_scale;
  p.batch = a->batch, p.n_rows = a->n_rows, p.c = a->c, p.m = a->m, p.first_block = a->first_block;
  p.out_batch_stride = a->out_batch_stride > 0 ? a->out_batch_stride : n_out;
  p.n_out = n_out;
  p.skip = (a->overlap && a->first_block > 0) ? 1 : 0;
  p.overlap = a->overlap;
  p.R = 1;
  if (n_out == 0 || p.batch == 0) return cudaSuccess;
  if (p.batch * n_out >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  if (a->in_dtype == HYB_F32) return launch_t<float>(p, a->out_dtype, s);
  return launch_t<__nv_bfloat16>(p, a->out_dtype, s);
}

}  // namespace hyb
