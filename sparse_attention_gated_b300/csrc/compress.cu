// compress.cu -- softmax-gated compressor ("DeepSeek-V4 hybrid attention"
// (trishampatil.com) section V.1 for CSA with overlap, section VI for HCA).
//
// One warp per (batch, output entry).  Lane l owns channels [l*V, l*V+V) with
// V = c/32, so every row of every input is read by one coalesced warp-wide
// load of c elements.  For each channel the kernel keeps an online softmax
// (running max, denominator, weighted numerator) over the window rows, in
// float32 and in base 2.  This kernel is HBM-bound: it reads each of the four
// inputs once (CSA rows are read by two neighbouring entries, stream a by
// entry i and stream b by entry i+1) and writes the entries once.
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
};

template <typename Tin, int V>
__device__ __forceinline__ void gate_accumulate(const Tin* __restrict__ zrow, const Tin* __restrict__ crow,
                                                const float* __restrict__ brow, float (&mx)[V], float (&den)[V],
                                                float (&num)[V]) {
  float z[V], cv[V], bv[V];
  load_vec<V>(zrow, z);
  load_vec<V>(crow, cv);
  load_vec<V>(brow, bv);
#pragma unroll
  for (int i = 0; i < V; ++i) {
    float l = (z[i] + bv[i]) * kLog2e;
    if (l > mx[i]) {
      float r = exp2f(mx[i] - l);  // 0 when mx = -inf
      den[i] = den[i] * r + 1.0f;
      num[i] = num[i] * r + cv[i];
      mx[i] = l;
    } else {
      float e = exp2f(l - mx[i]);
      den[i] += e;
      num[i] += e * cv[i];
    }
  }
}

// OUT: 0 = float32, 1 = bf16, 2 = e4m3 + per-entry scale
template <typename Tin, int V, int OUT>
__global__ void __launch_bounds__(256) compress_kernel(CompressParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= p.batch * p.n_out) return;
  const int64_t b = gw / p.n_out, j = gw % p.n_out;
  const int64_t lb = j + p.skip;
  const int64_t abs_blk = p.first_block + lb;
  const int64_t m = p.m, c = p.c;
  const int64_t ch0 = (int64_t)lane * V;

  float mx[V], den[V], num[V];
#pragma unroll
  for (int i = 0; i < V; ++i) mx[i] = -INFINITY, den[i] = 0.f, num[i] = 0.f;

  const Tin* ca = static_cast<const Tin*>(p.ca);
  const Tin* za = static_cast<const Tin*>(p.za);
  const int64_t base = b * p.n_rows;
  if (p.overlap && abs_blk > 0) {
    const Tin* cb = static_cast<const Tin*>(p.cb);
    const Tin* zb = static_cast<const Tin*>(p.zb);
    for (int64_t q = 0; q < m; ++q) {
      const int64_t row = base + (lb - 1) * m + q;
      gate_accumulate<Tin, V>(zb + row * c + ch0, cb + row * c + ch0, p.bias + q * c + ch0, mx, den, num);
    }
  }
  const int64_t pos0 = p.overlap ? m : 0;
  for (int64_t q = 0; q < m; ++q) {
    const int64_t row = base + lb * m + q;
    gate_accumulate<Tin, V>(za + row * c + ch0, ca + row * c + ch0, p.bias + (pos0 + q) * c + ch0, mx, den, num);
  }

  float r[V];
#pragma unroll
  for (int i = 0; i < V; ++i) r[i] = num[i] / den[i];

  const int64_t orow = b * p.out_batch_stride + j;
  if constexpr (OUT == 0) {
    store_vec<V>(static_cast<float*>(p.out) + orow * c + ch0, r);
  } else if constexpr (OUT == 1) {
    store_vec<V>(static_cast<__nv_bfloat16*>(p.out) + orow * c + ch0, r);
  } else {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) amax = fmaxf(amax, fabsf(r[i]));
    amax = warp_max(amax);
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint8_t codes[V];
#pragma unroll
    for (int i = 0; i < V; ++i)
      codes[i] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(r[i], scale), __NV_SATFINITE, __NV_E4M3);
    uint8_t* dst = static_cast<uint8_t*>(p.out) + orow * c + ch0;
#pragma unroll
    for (int i = 0; i < V; ++i) dst[i] = codes[i];
    if (lane == 0) p.out_scale[orow] = scale;
  }
}

template <typename Tin, int V>
static cudaError_t launch_v(const CompressParams& p, int out_dtype, cudaStream_t s) {
  const int64_t warps = p.batch * p.n_out;
  const int wpb = 8;
  const dim3 grid((unsigned)((warps + wpb - 1) / wpb)), block(32 * wpb);
  if (out_dtype == HYB_F32)
    compress_kernel<Tin, V, 0><<<grid, block, 0, s>>>(p);
  else if (out_dtype == HYB_BF16)
    compress_kernel<Tin, V, 1><<<grid, block, 0, s>>>(p);
  else
    compress_kernel<Tin, V, 2><<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_t(const CompressParams& p, int out_dtype, cudaStream_t s) {
  switch (p.c / 32) {
    case 1: return launch_v<Tin, 1>(p, out_dtype, s);
    case 2: return launch_v<Tin, 2>(p, out_dtype, s);
    case 4: return launch_v<Tin, 4>(p, out_dtype, s);
    case 8: return launch_v<Tin, 8>(p, out_dtype, s);
    case 16: return launch_v<Tin, 16>(p, out_dtype, s);
  }
  return cudaErrorInvalidValue;
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
  if (n_out == 0 || p.batch == 0) return cudaSuccess;
  if (a->in_dtype == HYB_F32) return launch_t<float>(p, a->out_dtype, s);
  return launch_t<__nv_bfloat16>(p, a->out_dtype, s);
}

}  // namespace hyb
