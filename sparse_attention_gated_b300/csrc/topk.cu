// topk.cu -- top-k selector of the lightning indexer ("DeepSeek-V4 hybrid
// attention" (trishampatil.com) section V.2: the k best-scoring compressed
// blocks are kept; "DeepSeek-V4: Anatomy..." (modernaiengineering.com) worked
// example: fewer than k entries are kept when fewer exist).
//
// One CTA of 1024 threads per query row.  Exact radix select on the
// order-preserving uint32 image of the float32 scores, 8 bits per pass from
// the top: after four passes the threshold key T (the k-th largest) and the
// number of ties to keep are known.  The kept set is every entry with key > T
// plus the lowest-indexed entries with key == T, i.e. ranking by
// (score descending, index ascending).  It is written in ascending index
// order (a bitonic sort in shared memory) and padded with -1.
// Rows that fit (<= kStageCap scores) are staged once in shared memory;
// longer rows (decode over 10^5 entries) are re-read from L2 on each pass.
#include "kernels.cuh"

namespace hyb {

constexpr int kTopkThreads = 1024;
constexpr int64_t kStageCap = 16384;

struct TopkParams {
  const float* scores;
  int64_t score_stride;
  int32_t* idx;
  float* out_scores;
  int64_t n_q, n_entries, m, k, q_pos0, kp;
};

template <bool STAGED>
__device__ __forceinline__ uint32_t row_key(const uint32_t* keys_s, const float* sc, int64_t s) {
  if constexpr (STAGED)
    return keys_s[s];
  else
    return float_order_key(__ldg(sc + s));
}

// append to the selection; never writes past its kp slots
__device__ __forceinline__ void push_sel(int32_t* sel, int* n, int64_t kp, int32_t s) {
  const int pos = atomicAdd(n, 1);
  if (pos < kp) sel[pos] = s;
}

template <bool STAGED>
__global__ void __launch_bounds__(kTopkThreads) topk_radix_kernel(TopkParams p) {
  extern __shared__ uint32_t dyn[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_prefix, s_mask, s_desired, s_chunk_eq;
  __shared__ int s_nsel;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t j = row % p.n_q;
  int64_t vis = visible_entries(p.q_pos0 + j, p.m);
  if (vis > p.n_entries) vis = p.n_entries;
  const float* sc = p.scores + row * p.score_stride;
  int32_t* out = p.idx + row * p.k;
  float* out_sc = p.out_scores ? p.out_scores + row * p.k : nullptr;

  if (vis <= p.k) {  // everything visible is kept, already in ascending order
    for (int64_t i = tid; i < p.k; i += kTopkThreads) {
      out[i] = i < vis ? (int32_t)i : -1;
      if (out_sc) out_sc[i] = i < vis ? sc[i] : -INFINITY;
    }
    return;
  }

  uint32_t* keys_s = dyn;                                                  // [vis] when STAGED
  int32_t* sel = reinterpret_cast<int32_t*>(dyn + (STAGED ? kStageCap : 0));  // [kp]
  if constexpr (STAGED) {
    for (int64_t s = tid; s < vis; s += kTopkThreads) keys_s[s] = float_order_key(__ldg(sc + s));
  }
  if (tid == 0) s_prefix = 0, s_mask = 0, s_desired = (uint32_t)p.k, s_nsel = 0;
  __syncthreads();

  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int64_t s = tid; s < vis; s += kTopkThreads) {
      const uint32_t key = row_key<STAGED>(keys_s, sc, s);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l covers digits hi..hi-7 with hi = 255 - 8l (lane 0 = largest digits)
      const int hi = 255 - 8 * lane;
      uint32_t lane_sum = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) lane_sum += hist[hi - d];
      uint32_t incl = lane_sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - lane_sum;
      const uint32_t desired = s_desired;
      if (excl < desired && desired <= incl) {
        uint32_t cum = excl;
        for (int d = hi; d > hi - 8; --d) {
          if (cum + hist[d] >= desired) {
            s_prefix = prefix | ((uint32_t)d << shift);
            s_mask = mask | (255u << shift);
            s_desired = desired - cum;
            break;
          }
          cum += hist[d];
        }
      }
    }
    __syncthreads();
  }

  const uint32_t T = s_prefix;
  const uint32_t ties = s_desired;  // how many entries with key == T to keep (the lowest indices)
  uint32_t eq_base = 0;
  for (int64_t base = 0; base < vis; base += kTopkThreads) {
    const int64_t s = base + tid;
    const uint32_t key = s < vis ? row_key<STAGED>(keys_s, sc, s) : 0u;
    const bool gt = s < vis && key > T;
    const bool eq = s < vis && key == T;
    if (gt) push_sel(sel, &s_nsel, p.kp, (int32_t)s);
    const uint32_t ball = __ballot_sync(0xffffffffu, eq);
    const uint32_t lane_rank = __popc(ball & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(ball);
    __syncthreads();
    if (warp == 0) {
      const uint32_t v = warp_tot[lane];
      uint32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      warp_tot[lane] = incl - v;  // exclusive offset of each warp
      if (lane == 31) s_chunk_eq = incl;
    }
    __syncthreads();
    if (eq && eq_base + warp_tot[warp] + lane_rank < ties) push_sel(sel, &s_nsel, p.kp, (int32_t)s);
    eq_base += s_chunk_eq;
    __syncthreads();
    if (eq_base >= ties && base + kTopkThreads < vis) {
      // all ties taken; the remaining chunks can only add entries with key > T
      for (int64_t s2 = base + kTopkThreads + tid; s2 < vis; s2 += kTopkThreads) {
        if (row_key<STAGED>(keys_s, sc, s2) > T) push_sel(sel, &s_nsel, p.kp, (int32_t)s2);
      }
      break;
    }
  }
  for (int64_t i = p.k + tid; i < p.kp; i += kTopkThreads) sel[i] = INT32_MAX;
  __syncthreads();

  // bitonic sort of sel[0..kp) ascending
  for (int64_t size = 2; size <= p.kp; size <<= 1) {
    for (int64_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (int64_t i = tid; i < p.kp; i += kTopkThreads) {
        const int64_t partner = i ^ stride;
        if (partner > i) {
          const bool up = (i & size) == 0;
          const int32_t a = sel[i], b = sel[partner];
          if ((a > b) == up) sel[i] = b, sel[partner] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int64_t i = tid; i < p.k; i += kTopkThreads) {
    out[i] = sel[i];
    if (out_sc) out_sc[i] = sc[sel[i]];
  }
}

size_t topk_workspace_bytes(const hyb_index_args*, int64_t) { return 0; }

cudaError_t launch_topk(const hyb_index_args* a, const float* scores, int64_t score_stride, void*, cudaStream_t s) {
  TopkParams p;
  p.scores = scores, p.score_stride = score_stride, p.idx = a->idx, p.out_scores = a->scores;
  p.n_q = a->n_q, p.n_entries = a->n_entries, p.m = a->m, p.k = a->k, p.q_pos0 = a->q_pos0;
  int64_t kp = 1;
  while (kp < a->k) kp <<= 1;
  p.kp = kp;
  const int64_t rows = a->batch * a->n_q;
  if (rows == 0) return cudaSuccess;
  const int64_t n_vis_max = std::min<int64_t>(visible_entries(a->q_pos0 + a->n_q - 1, a->m), a->n_entries);
  if (n_vis_max <= kStageCap) {
    const size_t smem = sizeof(uint32_t) * (size_t)kStageCap + sizeof(int32_t) * (size_t)kp;
    cudaFuncSetAttribute(topk_radix_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    topk_radix_kernel<true><<<(unsigned)rows, kTopkThreads, smem, s>>>(p);
  } else {
    const size_t smem = sizeof(int32_t) * (size_t)kp;
    cudaFuncSetAttribute(topk_radix_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    topk_radix_kernel<false><<<(unsigned)rows, kTopkThreads, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace hyb
