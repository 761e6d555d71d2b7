// compress.cu -- softmax-gated compressor ("DeepSeek-V4 hybrid attention"
// (trishampatil.com) section V.1 for CSA with overlap, section VI for HCA).
//
// For entry i and channel ch the gate is a softmax over the W rows of the
// entry's window (W = 2m with overlap, m without) of Z[row][ch] + bias[pos][ch],
// and the entry is the gate-weighted sum of C[row][ch].
//
// Work decomposition: one CTA per (entry, slab of S channels).  S starts at c
// and halves (down to 16) until there are at least two CTAs per SM, so a
// decode step that compresses only a handful of entries still spreads over
// the whole GPU.  Inside a CTA, G = S/4 channel threads (4 channels each: one
// 8-byte bf16 / 16-byte f32 load per row) times R row groups (a power of two);
// row group g takes window rows g, g+R, ...  A thread loads up to 4 of its rows
// at once, takes their maximum per channel, then accumulates the denominator
// and the weighted numerator relative to its running maximum (base 2, float32).
// The R partial states (max, denominator, numerator) are merged by a tree in
// shared memory.  E4M3 output needs the whole entry for its scale (amax/448),
// so it keeps S = c; so does MXFP4 output (a scale per block of 32 channels).
//
// A batch of up to kCompressBatchMax compressions (the entries that complete at one decode
// step in the CSA layer, its indexer keys and the HCA layer) runs as one launch: CTA
// ranges per call, 256 threads, each call with its own S and R.
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
  int64_t batch, n_rows, in_batch_stride, c, m, first_block, out_batch_stride, n_out, skip;
  int overlap;
  int S;  // channels per CTA
  int R;  // row groups (power of two)
};

constexpr int kCv = 4;           // channels per thread
constexpr int kRowBatch = 4;     // rows loaded at once per thread
constexpr int kCompressThreads = 256;

// e2m1 code of a float32 (OCP microscaling FP4): the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6,
// a tie going to the code with an even last bit, above 6 saturated; bit 3 the sign.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t m = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                   : a <= 2.5f ? 4u : a < 3.5f ? 5u : a <= 5.0f ? 6u : 7u;
  return m | ((__float_as_uint(y) >> 31) << 3);
}

// One CTA's work: entry bj of the call (b * n_out + j), channel slab `slab`.  OUT: 0 =
// float32, 1 = bf16, 2 = e4m3 + per-entry scale, 3 = MXFP4 (e2m1 codes two per byte +
// an e8m0 scale byte per 32 channels).  Threads past the call's G x R (a batch
// launch sizes its CTAs for the largest call) accumulate nothing.
template <typename Tin, int OUT>
__device__ __forceinline__ void compress_cta(const CompressParams& p, int64_t bj, int64_t slab, float* sm,
                                             float* s_red) {
  const int64_t c = p.c, m = p.m;
  const int G = p.S / kCv;
  const int g = threadIdx.x % G, rg = threadIdx.x / G;
  const bool live = rg < p.R;
  const int64_t b = bj / p.n_out, j = bj % p.n_out;
  const int64_t lb = j + p.skip;  // block index within the rows passed in
  const bool has_prev = p.overlap && p.first_block + lb > 0;
  const int64_t ch0 = slab * p.S + g * kCv;
  const int W = (int)(p.overlap ? 2 * m : m);
  const int64_t base = b * p.in_batch_stride;
  const Tin* ca = static_cast<const Tin*>(p.ca);
  const Tin* za = static_cast<const Tin*>(p.za);
  const Tin* cb = static_cast<const Tin*>(p.cb);
  const Tin* zb = static_cast<const Tin*>(p.zb);

  float mx[kCv], den[kCv], num[kCv];
#pragma unroll
  for (int i = 0; i < kCv; ++i) mx[i] = -INFINITY, den[i] = 0.f, num[i] = 0.f;

  for (int pos0 = rg; live && pos0 < W; pos0 += kRowBatch * p.R) {
    float lg[kRowBatch][kCv], cv[kRowBatch][kCv];
    bool have[kRowBatch];
#pragma unroll
    for (int u = 0; u < kRowBatch; ++u) {
      const int pos = pos0 + u * p.R;
      // window position pos: stream b over block lb-1 for pos < m (overlap), else stream a over block lb
      const bool prev = p.overlap && pos < m;
      have[u] = pos < W && (!prev || has_prev);
      float z[kCv], bv[kCv];
      if (have[u]) {
        const int64_t row = base + (prev ? (lb - 1) * m + pos : lb * m + (p.overlap ? pos - m : pos));
        load_vec<kCv>((prev ? zb : za) + row * c + ch0, z);
        load_vec<kCv>((prev ? cb : ca) + row * c + ch0, cv[u]);
        load_vec<kCv>(p.bias + (int64_t)pos * c + ch0, bv);
#pragma unroll
        for (int i = 0; i < kCv; ++i) lg[u][i] = (z[i] + bv[i]) * kLog2e;
      } else {
#pragma unroll
        for (int i = 0; i < kCv; ++i) lg[u][i] = -INFINITY, cv[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < kCv; ++i) {
      float bm = mx[i];
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u) bm = fmaxf(bm, lg[u][i]);
      if (bm == -INFINITY) continue;  // nothing in this batch or before
      const float r = exp2f(mx[i] - bm);  // 0 when mx = -inf
      float d = den[i] * r, n = num[i] * r;
#pragma unroll
      for (int u = 0; u < kRowBatch; ++u) {
        const float e = exp2f(lg[u][i] - bm);  // 0 for absent rows
        d += e;
        n = fmaf(e, cv[u][i], n);
      }
      mx[i] = bm, den[i] = d, num[i] = n;
    }
  }

  // tree merge of the R row-group states
  float* s_mx = sm;
  float* s_den = sm + p.R * p.S;
  float* s_num = s_den + p.R * p.S;
  const int lo = g * kCv;
  for (int half = p.R >> 1; half >= 1; half >>= 1) {
    if (rg >= half && rg < 2 * half) {
      const int o = (rg - half) * p.S + lo;
#pragma unroll
      for (int i = 0; i < kCv; ++i) s_mx[o + i] = mx[i], s_den[o + i] = den[i], s_num[o + i] = num[i];
    }
    __syncthreads();
    if (rg < half) {
      const int o = rg * p.S + lo;
#pragma unroll
      for (int i = 0; i < kCv; ++i) {
        const float m2 = s_mx[o + i];
        const float M = fmaxf(mx[i], m2);
        if (M == -INFINITY) continue;
        const float f1 = exp2f(mx[i] - M), f2 = exp2f(m2 - M);
        den[i] = den[i] * f1 + s_den[o + i] * f2;
        num[i] = num[i] * f1 + s_num[o + i] * f2;
        mx[i] = M;
      }
    }
    __syncthreads();
  }

  float r[kCv];
#pragma unroll
  for (int i = 0; i < kCv; ++i) r[i] = num[i] / den[i];
  const int64_t orow = b * p.out_batch_stride + j;
  if constexpr (OUT == 0) {
    if (rg == 0) store_vec<kCv>(static_cast<float*>(p.out) + orow * c + ch0, r);
  } else if constexpr (OUT == 1) {
    if (rg == 0) store_vec<kCv>(static_cast<__nv_bfloat16*>(p.out) + orow * c + ch0, r);
  } else if constexpr (OUT == 3) {
    // per block of 32 channels (8 consecutive channel threads of one warp): E = floor(log2
    // amax) - 2 clamped to [-127, 127] (-127 for amax = 0; floor(log2) of a float32 is its
    // unbiased exponent field, which already lies below -127 for subnormals), scale byte
    // E + 127, codes of value * 2^-E (exact scaling by a power of two)
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kCv; ++i) amax = fmaxf(amax, fabsf(r[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int E = -127;
    if (amax > 0.f) E = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 2;
    E = E < -127 ? -127 : (E > 127 ? 127 : E);
    if (rg == 0) {
      // 2^-E as a float32: E in [-127, 127] gives exponents 0..254; 2^127 (E = -127) is
      // 0x7F000000, and every factor is a normal power of two
      const float inv = __uint_as_float((uint32_t)(127 - E) << 23);
      uint32_t packed = 0;
#pragma unroll
      for (int i = 0; i < kCv; ++i) packed |= e2m1_code(r[i] * inv) << (4 * i);
      *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(p.out) + orow * (c / 2) + ch0 / 2) = (uint16_t)packed;
      if ((ch0 & 31) == 0)
        reinterpret_cast<uint8_t*>(p.out_scale)[orow * (c / 32) + ch0 / 32] = (uint8_t)(E + 127);
    }
  } else {
    // per-entry scale = amax / 448 over all c channels (this CTA holds the whole entry)
    float amax = 0.f;
    if (rg == 0)
#pragma unroll
      for (int i = 0; i < kCv; ++i) amax = fmaxf(amax, fabsf(r[i]));
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_red[w]);
    if (rg == 0) {
      const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      uint32_t codes = 0;
#pragma unroll
      for (int i = 0; i < kCv; ++i)
        codes |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(r[i], scale), __NV_SATFINITE, __NV_E4M3) << (8 * i);
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.out) + orow * c + ch0) = codes;
      if (threadIdx.x == 0) p.out_scale[orow] = scale;
    }
  }
}

template <typename Tin, int OUT>
__global__ void __launch_bounds__(kCompressThreads) compress_kernel(CompressParams p) {
  extern __shared__ float sm[];  // [3][R][S]: max, denominator, numerator of each row group
  __shared__ float s_red[kCompressThreads / 32];
  pdl_wait();
  pdl_trigger();
  compress_cta<Tin, OUT>(p, blockIdx.x, blockIdx.y, sm, s_red);
}

struct CompressBatch {
  CompressParams call[kCompressBatchMax];
  int out[kCompressBatchMax];        // OUT of each call
  int64_t cta_end[kCompressBatchMax];  // CTAs of calls 0..i
  int64_t slabs[kCompressBatchMax];    // c / S of each call
  int n;
};

template <typename Tin>
__global__ void __launch_bounds__(kCompressThreads) compress_batch_kernel(const __grid_constant__ CompressBatch B) {
  extern __shared__ float sm[];
  __shared__ float s_red[kCompressThreads / 32];
  pdl_wait();
  pdl_trigger();
  int i = 0;
  while (i + 1 < B.n && (int64_t)blockIdx.x >= B.cta_end[i]) ++i;
  const int64_t local = (int64_t)blockIdx.x - (i ? B.cta_end[i - 1] : 0);
  const int64_t bj = local / B.slabs[i], slab = local % B.slabs[i];
  switch (B.out[i]) {  // (the same for every thread of the CTA)
    case 0: compress_cta<Tin, 0>(B.call[i], bj, slab, sm, s_red); break;
    case 1: compress_cta<Tin, 1>(B.call[i], bj, slab, sm, s_red); break;
    case 2: compress_cta<Tin, 2>(B.call[i], bj, slab, sm, s_red); break;
    default: compress_cta<Tin, 3>(B.call[i], bj, slab, sm, s_red); break;
  }
}

// S and R of one call: S halves (from c, down to 16) until the call has at least two CTAs
// per SM (e4m3 output keeps the whole entry in one CTA); R doubles while it fits.
static void shape_call(CompressParams& p, int out_dtype) {
  const int W = (int)(p.overlap ? 2 * p.m : p.m);
  int S = (int)p.c;
  if (out_dtype != HYB_E4M3 && out_dtype != HYB_MXFP4)
    while (S > 16 && p.batch * p.n_out * (p.c / S) < 2 * kNumSMs) S >>= 1;
  const int G = S / kCv;
  int R = 1;
  while (2 * R <= W && 2 * R * G <= kCompressThreads) R <<= 1;
  p.S = S, p.R = R;
}

template <typename Tin>
static cudaError_t launch_t(CompressParams& p, int out_dtype, cudaStream_t s) {
  shape_call(p, out_dtype);
  const int S = p.S, R = p.R, G = S / kCv;
  const size_t smem = (size_t)3 * R * S * sizeof(float);
  const dim3 grid((unsigned)(p.batch * p.n_out), (unsigned)(p.c / S)), block((unsigned)(G * R));
  cudaError_t e;
  if (out_dtype == HYB_F32) {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = launch_pdl(compress_kernel<Tin, 0>, grid, block, smem, s, p);
  } else if (out_dtype == HYB_BF16) {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = launch_pdl(compress_kernel<Tin, 1>, grid, block, smem, s, p);
  } else if (out_dtype == HYB_E4M3) {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = launch_pdl(compress_kernel<Tin, 2>, grid, block, smem, s, p);
  } else {
    e = cudaFuncSetAttribute(compress_kernel<Tin, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = launch_pdl(compress_kernel<Tin, 3>, grid, block, smem, s, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool compress_shape_supported(int64_t c) { return c == 32 || c == 64 || c == 128 || c == 256 || c == 512; }

static CompressParams make_params(const hyb_compress_args* a, int64_t n_out) {
  CompressParams p;
  p.ca = a->ca, p.cb = a->cb, p.za = a->za, p.zb = a->zb, p.bias = a->bias, p.out = a->out, p.out_scale = a->out_scale;
  p.batch = a->batch, p.n_rows = a->n_rows, p.c = a->c, p.m = a->m, p.first_block = a->first_block;
  p.in_batch_stride = a->in_batch_stride > 0 ? a->in_batch_stride : a->n_rows;
  p.out_batch_stride = a->out_batch_stride > 0 ? a->out_batch_stride : n_out;
  p.n_out = n_out;
  p.skip = (a->overlap && a->first_block > 0) ? 1 : 0;
  p.overlap = a->overlap;
  p.S = (int)a->c, p.R = 1;
  return p;
}

cudaError_t launch_compress(const hyb_compress_args* a, int64_t n_out, cudaStream_t s) {
  CompressParams p = make_params(a, n_out);
  if (n_out == 0 || p.batch == 0) return cudaSuccess;
  if (p.batch * n_out >= (int64_t(1) << 31) - 1) return cudaErrorInvalidConfiguration;
  if (a->in_dtype == HYB_F32) return launch_t<float>(p, a->out_dtype, s);
  return launch_t<__nv_bfloat16>(p, a->out_dtype, s);
}

// calls with no output are left out; all calls have the same input type (checked by the caller)
cudaError_t launch_compress_batch(const hyb_compress_args* const* a, const int64_t* n_out, int n, cudaStream_t s) {
  CompressBatch B{};
  size_t smem = 0;
  int64_t ctas = 0;
  for (int i = 0; i < n; ++i) {
    if (n_out[i] == 0 || a[i]->batch == 0) continue;
    CompressParams p = make_params(a[i], n_out[i]);
    if (p.batch * n_out[i] >= (int64_t(1) << 31) - 1) return cudaErrorInvalidConfiguration;
    shape_call(p, a[i]->out_dtype);
    const int k = B.n++;
    B.call[k] = p;
    B.out[k] = a[i]->out_dtype == HYB_F32 ? 0 : a[i]->out_dtype == HYB_BF16 ? 1 : a[i]->out_dtype == HYB_E4M3 ? 2 : 3;
    B.slabs[k] = p.c / p.S;
    ctas += p.batch * n_out[i] * B.slabs[k];
    B.cta_end[k] = ctas;
    smem = std::max(smem, (size_t)3 * p.R * p.S * sizeof(float));
  }
  if (B.n == 0) return cudaSuccess;
  if (ctas >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  const bool f32 = a[0]->in_dtype == HYB_F32;
  cudaError_t e = f32 ? cudaFuncSetAttribute(compress_batch_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                      : cudaFuncSetAttribute(compress_batch_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = f32 ? launch_pdl(compress_batch_kernel<float>, dim3((unsigned)ctas), dim3(kCompressThreads), smem, s, B)
          : launch_pdl(compress_batch_kernel<__nv_bfloat16>, dim3((unsigned)ctas), dim3(kCompressThreads), smem, s, B);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
