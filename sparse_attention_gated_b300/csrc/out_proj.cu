// out_proj.cu -- grouped output projection on the 5th-generation tensor cores ("DeepSeek-V4
// hybrid attention" (trishampatil.com) section V.3, core attention and grouped output: the
// heads are split into g groups of n_h/g consecutive heads, each group's values are projected
// by a matrix of its own, and the g results are concatenated).
//
//   out[r, j*d_g + e] = sum_k W[j, e, k] * o[r, j*K + k],   K = (n_h/g) * c
//
// One CTA owns (group j, 128 consecutive output features e, up to N consecutive rows r) and
// accumulates the transposed tile out^T[e, r] in TMEM over the whole K:
//   D[e, r] += W_j[e, k-slab] . o_j[r, k-slab]^T      M = 128, N = 16..256 (rows), K = 64 per slab
// Both operands are K-major (W rows and o rows are contiguous in k), staged per 64-element
// slab by TMA in the 128-byte swizzle through a ring of stages.  At decode sizes (a few rows)
// the kernel streams the weights once (HBM-bound); with thousands of rows it is a GEMM whose
// operand tiles are reused from L2.  A single group (g = 1) is a plain projection, e.g. the
// concatenated result mapped to the model dimension.
//
// Warps: 0 TMA producer, 1 TMEM owner and MMA issuer, 2-5 epilogue (warp w reads TMEM lane
// quadrant w % 4: thread e of the four owns feature e0 + e and writes it for every row, so
// each row's 128 features are one coalesced store per warp group).  Every wait is bounded.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace hyb {

namespace {

constexpr int kM = 128;            // output features per CTA (MMA M)
constexpr int kSlabK = 64;         // K per stage (128 bytes of bf16)
constexpr int kASlab = kM * 128;   // 16 KiB of W per stage
constexpr int kThreads = 192;
constexpr int kRingBytes = 196 * 1024;

struct GpParams {
  void* out;
  int32_t out_bf16;
  int64_t rows, g, d_g, K;  // K = (n_h/g) * c, the inputs of one group
  int64_t out_stride;       // g * d_g
  int N;                    // rows per CTA (MMA N: 16, 32, ..., 256)
  int box_rows;             // rows of o per copy: N, or all the rows when there are fewer (the
                            // product's columns past them are never stored)
  int stages;
  int32_t* dev_status;
};

__global__ void __launch_bounds__(kThreads, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_o, GpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = kASlab + p.N * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + p.stages;
  uint64_t* done = empty + p.stages;
  volatile int* s_abort = reinterpret_cast<volatile int*>(done + 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work: (group, feature tile, row tile), row tile fastest so that CTAs sharing W run together
  const int64_t e_tiles = p.d_g / kM, r_tiles = (p.rows + p.N - 1) / p.N;
  const int64_t rt = blockIdx.x % r_tiles;
  const int64_t et = (blockIdx.x / r_tiles) % e_tiles;
  const int64_t j = blockIdx.x / (r_tiles * e_tiles);
  const int64_t row0 = rt * p.N, e0 = et * kM;
  const int64_t nk = p.K / kSlabK;
  uint32_t tmem_cols = 32;
  while ((int)tmem_cols < p.N) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) tc::mbar_init(&full[s], 1), tc::mbar_init(&empty[s], 1);
    tc::mbar_init(done, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(s_tmem, tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_w);
      tc::prefetch_tmap(&tm_o);
      int64_t last[16];
      for (int s = 0; s < 16; ++s) last[s] = -1;
      bool ok = true;
      for (int64_t kk = 0; kk < nk && ok; ++kk) {
        const int s = (int)(kk % p.stages);
        if (!(ok = tc::mbar_wait(&empty[s], (uint32_t)((kk / p.stages) & 1) ^ 1u, s_abort, 1))) break;
        uint8_t* st = smem + s * stage_bytes;
        tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(kASlab + p.box_rows * 128));
        tc::tma_load_2d(st, &tm_w, &full[s], (int32_t)(kk * kSlabK), (int32_t)(j * p.d_g + e0));
        tc::tma_load_2d(st + kASlab, &tm_o, &full[s], (int32_t)(j * p.K + kk * kSlabK), (int32_t)row0);
        if (s < 16) last[s] = kk;
      }
      if (!ok)
        for (int s = 0; s < p.stages && s < 16; ++s)
          if (last[s] >= 0) tc::mbar_wait_drain(&full[s], (uint32_t)((last[s] / p.stages) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (tc::elect_one()) {
      const uint32_t idesc = tc::make_idesc(1, 1, 0, 0, kM, (uint32_t)p.N);
      const uint32_t base = tc::smem_u32(smem);
      bool ok = true;
      for (int64_t kk = 0; kk < nk && ok; ++kk) {
        const int s = (int)(kk % p.stages);
        if (!(ok = tc::mbar_wait(&full[s], (uint32_t)((kk / p.stages) & 1), s_abort, 2))) break;
        tc::tc_fence_after();
        const uint32_t a = base + (uint32_t)(s * stage_bytes), b = a + kASlab;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tc::mma_f16(tmem, tc::desc_kmajor_sw128(a + 32 * q), tc::desc_kmajor_sw128(b + 32 * q), idesc,
                      (kk > 0 || q > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(done);  // completes once, after every product above
      tc::mbar_wait_drain(done, 0);
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int q4 = warp & 3;
    const int e = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    if (tc::mbar_wait(done, 0, s_abort, 3)) {
      tc::tc_fence_after();
      const int64_t col = j * p.d_g + e0 + e;
      for (int n0 = 0; n0 < p.N; n0 += 32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_base + (uint32_t)n0, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int64_t r = row0 + n0 + x;
          if (n0 + x < p.N && r < p.rows) {
            if (p.out_bf16)
              static_cast<__nv_bfloat16*>(p.out)[r * p.out_stride + col] = __float2bfloat16_rn(v[x]);
            else
              static_cast<float*>(p.out)[r * p.out_stride + col] = v[x];
          }
        }
      }
    }
  }
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT | ((*s_abort & 0xFF) << 8));
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

bool out_proj_shape_supported(int64_t n_h, int64_t c, int64_t g, int64_t d_g) {
  if (g < 1 || n_h % g != 0 || d_g % kM != 0) return false;
  const int64_t K = (n_h / g) * c;
  return K % kSlabK == 0 && K >= kSlabK;
}

cudaError_t launch_out_proj(const void* o, const void* w, void* out, int out_bf16, int64_t rows, int64_t n_h, int64_t c,
                            int64_t g, int64_t d_g, int64_t out_stride, int32_t* dev_status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  GpParams p{};
  p.out = out, p.out_bf16 = out_bf16, p.rows = rows, p.g = g, p.d_g = d_g, p.K = (n_h / g) * c;
  p.out_stride = out_stride;
  p.dev_status = dev_status;
  // rows per CTA: the smallest multiple of 16 that covers the rows, at most 256
  int N = (int)std::min<int64_t>(256, (rows + 15) / 16 * 16);
  p.N = N;
  const int stage_bytes = kASlab + N * 128;
  p.stages = std::min(16, kRingBytes / stage_bytes);
  // a copy of N rows past the last row reads zeros; with fewer rows than N the box holds them all
  p.box_rows = (int)std::min<int64_t>(N, rows);
  CUtensorMap tm_w, tm_o;
  if (!encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)p.K, (uint64_t)(g * d_g), (uint64_t)p.K * 2,
                      kSlabK, kM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o, (uint64_t)(n_h * c), (uint64_t)rows,
                      (uint64_t)(n_h * c) * 2, kSlabK, (uint32_t)p.box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t grid = g * (d_g / kM) * ((rows + N - 1) / N);
  if (grid >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)kRingBytes + (2 * 16 + 1) * 8 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(out_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(out_proj_kernel, dim3((unsigned)grid), dim3(kThreads), smem, s, tm_w, tm_o, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
