// sink.cu -- per-head attention sink ("DeepSeek-V4 hybrid attention"
// (trishampatil.com) section IV: a learnable sink per head inside both
// branches).
//
// The sink is one more logit s_h in a head's softmax denominator, with no
// value.  Because the branch's result is a log-sum-exp union, the sink can be
// added once to any stage's (o, lse): o *= exp(lse - L), lse = L with
// L = log(exp(lse) + exp(s_h)).  One warp per (query, head) row: lane 0's
// view of lse is read by every lane before lane 0 writes L; the lanes then
// scale the row's c values in place (float32 or bf16).
#include "kernels.cuh"

namespace hyb {

__global__ void __launch_bounds__(256) sink_kernel(void* out, int out_bf16, float* lse, const float* sink,
                                                   int64_t rows, int64_t n_h, int64_t c) {
  pdl_wait();
  pdl_trigger();
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float a = lse[r], s = sink[r % n_h];
  float L;
  if (a == -INFINITY && s == -INFINITY) {
    L = -INFINITY;
  } else {
    const float mx = fmaxf(a, s);
    L = mx + logf(expf(a - mx) + expf(s - mx));
  }
  const float f = a == -INFINITY ? 0.f : expf(a - L);
  __syncwarp();
  if (lane == 0) lse[r] = L;
  if (out_bf16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + r * c;
    for (int64_t d = lane; d < c; d += 32) o[d] = __float2bfloat16_rn(__bfloat162float(o[d]) * f);
  } else {
    float* o = static_cast<float*>(out) + r * c;
    for (int64_t d = lane; d < c; d += 32) o[d] *= f;
  }
}

cudaError_t launch_sink(void* out, int32_t out_dtype, float* lse, const float* sink, int64_t rows, int64_t n_h,
                        int64_t c, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;  // 8 warps of 256 threads, one row each
  if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e = launch_pdl(sink_kernel, dim3((unsigned)blocks), dim3(256), 0, s, out, out_dtype == HYB_BF16 ? 1 : 0,
                             lse, sink, rows, n_h, c);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
