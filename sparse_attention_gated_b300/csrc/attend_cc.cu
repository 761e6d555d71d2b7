// attend_cc.cu -- MQA core attention on CUDA cores, for the three entry
// sources of the hybrid-attention forward:
//   mode 0, CSA: the entries listed by the top-k selector ("DeepSeek-V4 hybrid
//           attention" (trishampatil.com) section V.3);
//   mode 1, HCA: every visible entry, s < floor((t+1)/m') (same page, section VI);
//   mode 2, sliding window: raw rows max(0,t-n_win+1)..t, merged with the
//           compressed branch by log-sum-exp ("DeepSeek-V4: Anatomy..."
//           (modernaiengineering.com), "One query in a CSA layer", steps 4-5).
//
// One warp per (batch, query, head).  Lane l holds dims [l*V, l*V+V) of the
// query, of each key/value row and of the output (V = c/32), so each row is
// one coalesced 32-lane load; warps of the same CTA are heads of the same
// query and read the same rows (L1 hits).  Online softmax in base 2 with
// float32 state.  For decode (few queries, long lists) the list is split
// across CTAs; each split writes an unnormalised partial (o, max, sum) and a
// combine kernel merges them.  This path serves the float32 configuration
// and any shape the tensor-core kernels do not cover.
#include "kernels.cuh"

namespace hyb {

struct AttendParams {
  AttendJob j;
  int n_split;
  float* part_o;   // [batch][n_q][n_split][n_h][c]
  float2* part_ml; // [batch][n_q][n_split][n_h]  (max, sum) in base 2
};

constexpr int kUnroll = 4;

template <typename T, int V, int MODE>
__global__ void __launch_bounds__(256) attend_cc_kernel(AttendParams P) {
  pdl_wait();
  pdl_trigger();
  const AttendJob& J = P.j;
  const int lane = threadIdx.x & 31;
  const int hpb = blockDim.x >> 5;
  const int64_t h = (int64_t)blockIdx.x * hpb + (threadIdx.x >> 5);
  const int64_t jq = blockIdx.y / P.n_split;
  const int sp = blockIdx.y % P.n_split;
  const int64_t b = blockIdx.z;
  if (h >= J.n_h) return;
  const int64_t t = query_pos(J.q_pos, J.q_pos0, b * J.n_q + jq, jq);
  const bool report = lane == 0 && sp == 0 && (threadIdx.x >> 5) == 0 && blockIdx.x == 0;
  const int64_t c = J.c;

  // the entry list of this query
  int64_t L;
  int64_t first_row = 0;  // MODE 1/2: row of list position 0
  const int32_t* list = nullptr;
  if constexpr (MODE == 0) {
    L = J.list_len;
    list = J.idx + (b * J.n_q + jq) * J.list_len;
  } else if constexpr (MODE == 1) {
    L = visible_checked(t, J.m, J.n_entries, J.dev_status, report);
  } else {
    const int64_t kvp = J.kv_pos0s ? __ldg(J.kv_pos0s + b) : J.kv_pos0;
    L = window_rows(t, J.n_win, kvp, J.n_entries, &first_row, J.dev_status, report);
  }
  const int64_t chunk = (L + P.n_split - 1) / P.n_split;
  const int64_t e_begin = (int64_t)sp * chunk;
  const int64_t e_end = e_begin + chunk < L ? e_begin + chunk : L;

  const T* Kb = static_cast<const T*>(J.k) + b * J.kv_stride * c + (int64_t)lane * V;
  const T* Vb = static_cast<const T*>(J.v) + b * J.kv_stride * c + (int64_t)lane * V;
  const bool alias = J.k == J.v;
  const int64_t qoff = ((b * J.n_q + jq) * J.n_h + h) * c + (int64_t)lane * V;

  float qf[V];
  load_vec<V>(static_cast<const T*>(J.q) + qoff, qf);
  const float qs = J.scale * kLog2e;
#pragma unroll
  for (int i = 0; i < V; ++i) qf[i] *= qs;

  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float mx = -INFINITY, l = 0.f;

  for (int64_t e0 = e_begin; e0 < e_end; e0 += kUnroll) {
    int64_t row[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = e0 + u;
      ok[u] = e < e_end;
      row[u] = 0;
      if (ok[u]) {
        if constexpr (MODE == 0) {
          const int32_t s = list[e];
          if (s < 0) {
            ok[u] = false;
          } else if (s >= J.n_entries) {
            ok[u] = false;
            if (lane == 0) flag_status(J.dev_status, HYB_DEV_BAD_INDEX);
          } else {
            row[u] = s;
          }
        } else {
          row[u] = first_row + e;
        }
      }
    }
    float kv[kUnroll][V];
    float sc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (ok[u]) {
        load_vec<V>(Kb + row[u] * c, kv[u]);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) kv[u][i] = 0.f;
      }
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) d = fmaf(qf[i], kv[u][i], d);
      sc[u] = d;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) sc[u] = warp_sum(sc[u]);
    float mnew = mx;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (ok[u]) mnew = fmaxf(mnew, sc[u]);
    if (mnew == -INFINITY) continue;  // nothing valid yet
    const float alpha = exp2f(mx - mnew);
    l *= alpha;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] *= alpha;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (!ok[u]) continue;
      const float pu = exp2f(sc[u] - mnew);
      l += pu;
      if (alias) {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(pu, kv[u][i], acc[i]);
      } else {
        float vv[V];
        load_vec<V>(Vb + row[u] * c, vv);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(pu, vv[i], acc[i]);
      }
    }
    mx = mnew;
  }

  if (P.n_split > 1) {
    const int64_t pidx = ((b * J.n_q + jq) * P.n_split + sp) * J.n_h + h;
    store_vec<V>(P.part_o + pidx * c + (int64_t)lane * V, acc);
    if (lane == 0) P.part_ml[pidx] = make_float2(mx, l);
    return;
  }

  const int64_t li = (b * J.n_q + jq) * J.n_h + h;
  if constexpr (MODE != 2) {
    float o[V];
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = acc[i] * inv;
    store_vec<V>(J.o + qoff, o);
    if (lane == 0) J.lse[li] = l > 0.f ? (mx + __log2f(l)) * kLn2 : -INFINITY;
  } else {
    // merge with the compressed branch: one softmax over the union
    const float lse_w = l > 0.f ? (mx + __log2f(l)) * kLn2 : -INFINITY;
    const float lse_c = J.lse_in ? J.lse_in[li] : -INFINITY;
    const float M = fmaxf(lse_w, lse_c);
    float wc = 0.f, ww = 0.f, Lse = -INFINITY;
    if (M != -INFINITY) {
      const float ec = lse_c == -INFINITY ? 0.f : expf(lse_c - M);
      const float ew = lse_w == -INFINITY ? 0.f : expf(lse_w - M);
      const float den = ec + ew;
      wc = ec / den;
      ww = ew / (den * (l > 0.f ? l : 1.f));  // window accumulator is unnormalised
      Lse = M + logf(den);
    }
    float oc[V];
    if (J.o_in && wc != 0.f) {
      load_vec<V>(J.o_in + qoff, oc);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) oc[i] = 0.f;
    }
    float r[V];
#pragma unroll
    for (int i = 0; i < V; ++i) r[i] = wc * oc[i] + ww * acc[i];
    if (J.out_bf16)
      store_vec<V>(static_cast<__nv_bfloat16*>(J.out) + qoff, r);
    else
      store_vec<V>(static_cast<float*>(J.out) + qoff, r);
    if (lane == 0 && J.lse) J.lse[li] = Lse;
  }
}

// Merge the split partials of one (batch, query, head): warp per head.
template <int V>
__global__ void __launch_bounds__(256) attend_combine_kernel(AttendParams P) {
  pdl_wait();
  pdl_trigger();
  const AttendJob& J = P.j;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= J.batch * J.n_q * J.n_h) return;
  const int64_t h = gw % J.n_h;
  const int64_t bq = gw / J.n_h;  // b * n_q + j
  float M = -INFINITY;
  for (int sp = 0; sp < P.n_split; ++sp) M = fmaxf(M, P.part_ml[(bq * P.n_split + sp) * J.n_h + h].x);
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float l = 0.f;
  if (M != -INFINITY) {
    for (int sp = 0; sp < P.n_split; ++sp) {
      const int64_t pidx = (bq * P.n_split + sp) * J.n_h + h;
      const float2 ml = P.part_ml[pidx];
      if (ml.x == -INFINITY) continue;
      const float wgt = exp2f(ml.x - M);
      l = fmaf(wgt, ml.y, l);
      float po[V];
      load_vec<V>(P.part_o + pidx * J.c + (int64_t)lane * V, po);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(wgt, po[i], acc[i]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] *= inv;
  store_vec<V>(J.o + (bq * J.n_h + h) * J.c + (int64_t)lane * V, acc);
  if (lane == 0) J.lse[bq * J.n_h + h] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
}

bool attend_cc_shape_supported(int64_t c, int64_t n_h) {
  return (c == 32 || c == 64 || c == 128 || c == 256 || c == 512) && n_h >= 1;
}

static int64_t list_len_max(const AttendJob& j) {
  if (j.mode == 0) return j.list_len;
  if (j.mode == 1)
    return j.q_pos ? j.n_entries : std::min<int64_t>(visible_entries(j.q_pos0 + j.n_q - 1, j.m), j.n_entries);
  return j.n_win;
}

int attend_cc_splits(const AttendJob& j) {
  if (j.mode == 2) return 1;
  const int64_t warps = j.batch * j.n_q * j.n_h;
  const int64_t target = 4LL * kNumSMs * 32;  // enough resident warps to cover HBM latency
  int64_t s = (target + warps - 1) / std::max<int64_t>(warps, 1);
  const int64_t L = list_len_max(j);
  s = std::min<int64_t>(s, std::max<int64_t>(1, L / 64));  // at least 64 entries per split
  s = std::min<int64_t>(s, 64);
  return (int)std::max<int64_t>(s, 1);
}

size_t attend_cc_workspace_bytes(const AttendJob& j) {
  const int s = attend_cc_splits(j);
  if (s <= 1) return 0;
  const size_t n = (size_t)(j.batch * j.n_q * s * j.n_h);
  return n * (size_t)j.c * sizeof(float) + n * sizeof(float2) + 256;
}

template <typename T, int V>
static cudaError_t launch_tv(const AttendParams& P, cudaStream_t s) {
  const AttendJob& J = P.j;
  const int hpb = (J.n_h % 8 == 0) ? 8 : (J.n_h % 4 == 0) ? 4 : (J.n_h % 2 == 0) ? 2 : 1;
  const dim3 grid((unsigned)(J.n_h / hpb), (unsigned)(J.n_q * P.n_split), (unsigned)J.batch), block(32 * hpb);
  cudaError_t e;
  if (J.mode == 0)
    e = launch_pdl(attend_cc_kernel<T, V, 0>, grid, block, 0, s, P);
  else if (J.mode == 1)
    e = launch_pdl(attend_cc_kernel<T, V, 1>, grid, block, 0, s, P);
  else
    e = launch_pdl(attend_cc_kernel<T, V, 2>, grid, block, 0, s, P);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || P.n_split == 1) return e;
  const int64_t warps = J.batch * J.n_q * J.n_h;
  if ((e = launch_pdl(attend_combine_kernel<V>, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, P)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_t(const AttendParams& P, cudaStream_t s) {
  switch (P.j.c / 32) {
    case 1: return launch_tv<T, 1>(P, s);
    case 2: return launch_tv<T, 2>(P, s);
    case 4: return launch_tv<T, 4>(P, s);
    case 8: return launch_tv<T, 8>(P, s);
    case 16: return launch_tv<T, 16>(P, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attend_cc(const AttendJob& j, void* ws, cudaStream_t s) {
  if (j.batch == 0 || j.n_q == 0 || j.n_h == 0) return cudaSuccess;
  AttendParams P;
  P.j = j;
  P.n_split = attend_cc_splits(j);
  P.part_o = nullptr;
  P.part_ml = nullptr;
  if (P.n_split > 1) {
    const size_t n = (size_t)(j.batch * j.n_q * P.n_split * j.n_h);
    P.part_o = static_cast<float*>(ws);
    P.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + n * (size_t)j.c * sizeof(float));
  }
  if (j.dtype == HYB_F32) return launch_t<float>(P, s);
  return launch_t<__nv_bfloat16>(P, s);
}

}  // namespace hyb
