// indexer_tc.cu -- lightning-indexer scores on the 5th-generation tensor cores
// ("DeepSeek-V4 hybrid attention" (trishampatil.com) section V.2; the indexer
// runs in FP8, "DeepSeek-V4: Anatomy..." (modernaiengineering.com) step 2):
//
//   I[t,s] = sum_h w[t,h] * ReLU( (qs[t,h] q8[t,h]) . (ks[s] k8[s]) )
//
// Per tile of 128 entries the FP8 products Q8 K8^T are one tcgen05.mma
// (kind::f8f6f4, M = 128 entries, N = NQ queries x 64 heads, K = c_I = 128 in
// four K=32 steps) accumulating in TMEM in float32.  The epilogue warps read
// the accumulator rows (one entry per thread), apply the scales, ReLU and the
// head weights, and write one float32 score per (query, entry).
//
// Roles (one CTA, persistent over work units = (query group, chunk of entry tiles)):
//   warp 0      TMA producer: key tiles (16 KiB, 128-byte swizzle) + their
//               scales into a ring of stages; the query group's FP8 rows.
//   warp 1      TMEM allocator and MMA issuer (one elected thread).
//   warps 2..   epilogue (TMEM -> registers -> scores).
// Key stages are released by tcgen05.commit when their MMAs complete; TMEM
// accumulators are double/quad-buffered so the epilogue of tile i overlaps
// the loads and MMAs of tiles i+1...  Every wait is bounded (about 1 s): on
// expiry the kernel raises HYB_DEV_TIMEOUT in dev_status, drains its own
// copies in flight, frees TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace hyb {

template <int NQ>
struct IdxTc {
  static constexpr int kTileE = 128;
  static constexpr int kHeads = 64;
  static constexpr int kN = NQ * kHeads;
  static constexpr int kStages = NQ == 1 ? 5 : 4;
  static constexpr int kAcc = NQ == 1 ? 4 : 2;
  static constexpr int kTmemCols = kAcc * kN;  // 256 or 512
  static constexpr int kEpiWarps = 8;
  // decode: two groups of four epilogue warps take alternate tiles; prefill: the two
  // groups share each tile (two queries each)
  static constexpr int kEpiGroups = NQ == 1 ? 2 : 1;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kScaleRing = kStages + kAcc;
  static constexpr int kKeyBytes = kTileE * 128;
  static constexpr int kScaleBytes = kTileE * 4;
  static constexpr int kQBytes = kN * 128;
  static constexpr int kOffKeys = 0;
  static constexpr int kOffQ = kOffKeys + kStages * kKeyBytes;
  static constexpr int kOffScales = kOffQ + 2 * kQBytes;
  static constexpr int kOffW = kOffScales + kScaleRing * kScaleBytes;  // 3 x float[NQ*64]: w*qs, w, qs
  static constexpr int kOffHist = kOffW + 3 * kN * 4;  // decode: row histogram of the scores' top bits
  static constexpr int kHistBytes = NQ == 1 ? kTopkHistBins * 2 : 0;  // 16-bit counters, two per word
  static constexpr int kOffBar = kOffHist + kHistBytes;
  static constexpr int kNumBars = 2 * kStages + 4 + 2 * kAcc + 2 * kScaleRing + 2;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + flags + alignment slack
};

struct IdxTcParams {
  const float* w;
  const float* qI_scale;
  float* scores;
  uint32_t* ghist;  // optional (one query per unit): [rows][kTopkHistBins] histogram of the score keys' top bits
  int64_t score_stride;
  int64_t n_q, n_entries, kv_stride, m, q_pos0;
  const int64_t* q_pos;  // optional per-query positions [batch * n_q] (read after the grid-dependency wait)
  int64_t groups_per_b, tiles_per_unit, units_per_group, n_units;
  int32_t* dev_status;
};

struct IdxUnit {
  int64_t b, j0, nq, tile_begin, tile_end;
};

template <int NQ>
__device__ __forceinline__ IdxUnit idx_unit(const IdxTcParams& p, int64_t u) {
  IdxUnit U;
  const int64_t g = u / p.units_per_group, chunk = u % p.units_per_group;
  U.b = g / p.groups_per_b;
  U.j0 = (g % p.groups_per_b) * NQ;
  U.nq = p.n_q - U.j0 < NQ ? p.n_q - U.j0 : NQ;
  // entries the unit's queries see: the last one's with consecutive positions, the
  // largest over them with per-query positions
  int64_t vis = 0;
  if (p.q_pos == nullptr) {
    vis = visible_checked(p.q_pos0 + U.j0 + U.nq - 1, p.m, p.n_entries, nullptr, false);
  } else {
    for (int64_t q = 0; q < U.nq; ++q) {
      const int64_t v = visible_checked(__ldg(p.q_pos + U.b * p.n_q + U.j0 + q), p.m, p.n_entries, nullptr, false);
      vis = v > vis ? v : vis;
    }
  }
  const int64_t tiles = (vis + 127) / 128;
  U.tile_begin = chunk * p.tiles_per_unit;
  U.tile_end = U.tile_begin + p.tiles_per_unit < tiles ? U.tile_begin + p.tiles_per_unit : tiles;
  return U;
}

template <int NQ>
__global__ void __launch_bounds__(IdxTc<NQ>::kThreads, NQ == 1 ? 2 : 1)
    index_tc_kernel(const __grid_constant__ CUtensorMap tm_keys, const __grid_constant__ CUtensorMap tm_scales,
                    const __grid_constant__ CUtensorMap tm_q, IdxTcParams p) {
  using C = IdxTc<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* keys = smem + C::kOffKeys;
  uint8_t* qbuf = smem + C::kOffQ;
  float* scales = reinterpret_cast<float*>(smem + C::kOffScales);
  float* w_c = reinterpret_cast<float*>(smem + C::kOffW);  // w*qs
  float* w_w = w_c + C::kN;                                 // w
  float* w_q = w_w + C::kN;                                 // qs
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* q_full = empty + C::kStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint64_t* acc_empty = acc_full + C::kAcc;
  uint64_t* sc_full = acc_empty + C::kAcc;
  uint64_t* sc_empty = sc_full + C::kScaleRing;
  uint64_t* done_bar = sc_empty + C::kScaleRing;
  uint64_t* epi_bar = done_bar + 1;  // epilogue-group sync (bounded)
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + C::kNumBars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::kNumBars) + 1;
  int* s_allpos = reinterpret_cast<int*>(bars + C::kNumBars) + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) tc::mbar_init(&full[i], 1), tc::mbar_init(&empty[i], 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&q_full[i], 1), tc::mbar_init(&q_empty[i], 1);
    for (int i = 0; i < C::kAcc; ++i)
      tc::mbar_init(&acc_full[i], 1), tc::mbar_init(&acc_empty[i], C::kEpiWarps / C::kEpiGroups);
    for (int i = 0; i < C::kScaleRing; ++i)
      tc::mbar_init(&sc_full[i], 1), tc::mbar_init(&sc_empty[i], C::kEpiWarps / C::kEpiGroups);
    tc::mbar_init(done_bar, 1);
    tc::mbar_init(epi_bar, C::kEpiWarps * 32);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(s_tmem, C::kTmemCols);
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_keys);
    tc::prefetch_tmap(&tm_scales);
    tc::prefetch_tmap(&tm_q);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  // the CTA's first unit, from the parameters alone (64-bit divisions): computed while
  // the previous kernel may still be running (with positions in device memory, after
  // the wait: the previous kernel may have written them)
  IdxUnit U_first;
  if (p.q_pos == nullptr) U_first = idx_unit<NQ>(p, blockIdx.x);
  pdl_wait();  // (the setup above touched only shared memory, TMEM and the parameters)
  pdl_trigger();
  if (p.q_pos != nullptr) U_first = idx_unit<NQ>(p, blockIdx.x);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (tc::elect_one()) {
      int stage = 0;
      uint32_t sphase = 0;
      int64_t q_count = 0, seq = 0, issued = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        const IdxUnit U = u == blockIdx.x ? U_first : idx_unit<NQ>(p, u);
        if (U.tile_begin >= U.tile_end) continue;
        // per tile: the keys first (the long HBM read), then, on a unit's first tile, its
        // queries, then the tile's scales
        bool q_todo = true;
        for (int64_t t = U.tile_begin; t < U.tile_end; ++t, ++seq) {
          if (!(ok = tc::mbar_wait(&empty[stage], sphase ^ 1u, s_abort))) break;
          tc::mbar_arrive_expect_tx(&full[stage], C::kKeyBytes);
          tc::tma_load_2d(keys + stage * C::kKeyBytes, &tm_keys, &full[stage], 0,
                          (int32_t)(U.b * p.kv_stride + t * C::kTileE));
          ++issued;
          if (++stage == C::kStages) stage = 0, sphase ^= 1u;
          if (q_todo) {
            const int qb = (int)(q_count & 1);
            if (!(ok = tc::mbar_wait(&q_empty[qb], (uint32_t)((q_count >> 1) & 1) ^ 1u, s_abort))) break;
            tc::mbar_arrive_expect_tx(&q_full[qb], C::kQBytes);
            tc::tma_load_2d(qbuf + qb * C::kQBytes, &tm_q, &q_full[qb], 0, (int32_t)((U.b * p.n_q + U.j0) * C::kHeads));
            ++q_count;
            q_todo = false;
          }
          const int r = (int)(seq % C::kScaleRing);
          if (!(ok = tc::mbar_wait(&sc_empty[r], (uint32_t)((seq / C::kScaleRing) & 1) ^ 1u, s_abort))) break;
          tc::mbar_arrive_expect_tx(&sc_full[r], C::kScaleBytes);
          tc::tma_load_2d(scales + r * C::kTileE, &tm_scales, &sc_full[r], (int32_t)(t * C::kTileE), (int32_t)U.b);
        }
      }
      if (!ok) {
        // drain this thread's copies in flight before the CTA can exit
        for (int64_t i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
          tc::mbar_wait_drain(&full[i % C::kStages], (uint32_t)((i / C::kStages) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (tc::elect_one()) {
      constexpr uint32_t idesc = tc::make_idesc(0, 0, 0, 0, 128, C::kN);
      int stage = 0, acc = 0;
      uint32_t sphase = 0, aphase = 0;
      int64_t q_count = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        const IdxUnit U = u == blockIdx.x ? U_first : idx_unit<NQ>(p, u);
        if (U.tile_begin >= U.tile_end) continue;
        const int qb = (int)(q_count & 1);
        if (!(ok = tc::mbar_wait(&q_full[qb], (uint32_t)((q_count >> 1) & 1), s_abort))) break;
        const uint32_t b_base = tc::smem_u32(qbuf + qb * C::kQBytes);
        for (int64_t t = U.tile_begin; t < U.tile_end; ++t) {
          if (!(ok = tc::mbar_wait(&acc_empty[acc], aphase ^ 1u, s_abort))) break;
          if (!(ok = tc::mbar_wait(&full[stage], sphase, s_abort))) break;
          tc::tc_fence_after();
          const uint32_t a_base = tc::smem_u32(keys + stage * C::kKeyBytes);
          const uint32_t d = tmem_base + (uint32_t)(acc * C::kN);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_f8f6f4(d, tc::desc_kmajor_sw128(a_base + 32 * k), tc::desc_kmajor_sw128(b_base + 32 * k), idesc,
                           k > 0 ? 1u : 0u);
          tc::mma_commit(&empty[stage]);
          tc::mma_commit(&acc_full[acc]);
          if (++stage == C::kStages) stage = 0, sphase ^= 1u;
          if (++acc == C::kAcc) acc = 0, aphase ^= 1u;
        }
        if (!ok) break;
        tc::mma_commit(&q_empty[qb]);
        ++q_count;
      }
      // every MMA issued above has completed once done_bar flips
      tc::mma_commit(done_bar);
      tc::mbar_wait_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0 .. kEpiWarps*32-1
    const int quad = warp & 3;        // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;  // NQ = 4: which queries this warp handles (two each); NQ = 1: tile parity
    constexpr int kQPerWarp = NQ == 1 ? 1 : 2;
    constexpr int kEpiThreads = C::kEpiWarps * 32;
    // the epilogue warps meet on an mbarrier (bounded), never on a hardware barrier
    uint32_t ephase = 0;
    auto esync = [&]() -> bool {
      tc::mbar_arrive(epi_bar);
      const bool r = tc::mbar_wait(epi_bar, ephase, s_abort);
      ephase ^= 1u;
      return r;
    };
    // decode: histogram of the score keys' top kTopkHistBits bits of the current row
    // (16-bit counters packed two per word: a unit holds fewer than 2^16 entries), added
    // into the row's global histogram when the row changes and at the end
    const bool do_hist = NQ == 1 && p.ghist != nullptr;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + C::kOffHist);
    int64_t hist_row = -1;
    if (do_hist)
      for (int i = et; i < kTopkHistBins / 2; i += kEpiThreads) hist[i] = 0;
    // each thread takes 8 consecutive words (16 bins), read as two 16-byte vectors
    static_assert(kTopkHistBins / 2 == 8 * kEpiThreads, "one 8-word slice of the histogram per epilogue thread");
    auto flush_hist = [&](bool clear) {
      uint4* h4 = reinterpret_cast<uint4*>(hist) + 2 * et;
      const uint4 a = h4[0], b = h4[1];
      const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t* g = p.ghist + hist_row * kTopkHistBins + 16 * et;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (v[i] & 0xFFFFu) atomicAdd(g + 2 * i, v[i] & 0xFFFFu);
        if (v[i] >> 16) atomicAdd(g + 2 * i + 1, v[i] >> 16);
      }
      if (clear) h4[0] = h4[1] = make_uint4(0u, 0u, 0u, 0u);
    };
    int64_t seq = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
      const IdxUnit U = u == blockIdx.x ? U_first : idx_unit<NQ>(p, u);
      if (U.tile_begin >= U.tile_end) continue;
      if (!(ok = esync())) break;  // everyone is done with the previous unit's tables
      if (do_hist && U.b * p.n_q + U.j0 != hist_row) {
        if (hist_row >= 0) flush_hist(true);
        hist_row = U.b * p.n_q + U.j0;
      }
      if (et == 0) *s_allpos = 1;
      if (!(ok = esync())) break;
      for (int i = et; i < C::kN; i += kEpiThreads) {
        const int jq = i / C::kHeads, h = i % C::kHeads;
        float wv = 0.f, qs = 1.f;
        if (jq < U.nq) {
          const int64_t off = ((U.b * p.n_q) + U.j0 + jq) * C::kHeads + h;
          wv = p.w[off];
          qs = p.qI_scale[off];
        }
        w_c[i] = wv * qs;
        w_w[i] = wv;
        w_q[i] = qs;
        if (!(qs > 0.f)) *s_allpos = 0;
      }
      if (!(ok = esync())) break;
      const bool allpos = *s_allpos != 0;
      // entries each of this warp's queries sees (a score past them is not written)
      int64_t vis_q[kQPerWarp];
#pragma unroll
      for (int qi = 0; qi < kQPerWarp; ++qi) {
        const int q = NQ == 1 ? 0 : 2 * half + qi;
        const int64_t row = U.b * p.n_q + U.j0 + q;
        vis_q[qi] = q < U.nq ? visible_checked(query_pos(p.q_pos, p.q_pos0, row, U.j0 + q), p.m, p.n_entries,
                                               p.dev_status, lane == 0 && U.tile_begin == 0)
                             : 0;
      }
      for (int64_t t = U.tile_begin; t < U.tile_end; ++t, ++seq) {
        if (NQ == 1 && (int)(seq & 1) != half) continue;  // the other group's tile
        const int r = (int)(seq % C::kScaleRing);
        const int acc = (int)(seq % C::kAcc);
        const uint32_t aphase = (uint32_t)((seq / C::kAcc) & 1);
        if (!(ok = tc::mbar_wait(&acc_full[acc], aphase, s_abort))) break;
        if (!(ok = tc::mbar_wait(&sc_full[r], (uint32_t)((seq / C::kScaleRing) & 1), s_abort))) break;
        tc::tc_fence_after();
        const int row = quad * 32 + lane;
        const int64_t s = t * C::kTileE + row;
        const float ks = scales[r * C::kTileE + row];
        float score[kQPerWarp];
#pragma unroll
        for (int qi = 0; qi < kQPerWarp; ++qi) {
          const int q = NQ == 1 ? 0 : 2 * half + qi;
          const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * C::kN + q * C::kHeads);
          // heads 0-31 then 32-63 (one 32-column load live at a time), summed in four
          // interleaved partial sums (head h into sum h mod 4) that are then added pairwise
          const float* wc = w_c + q * C::kHeads;
          const float* ww = w_w + q * C::kHeads;
          const float* wq = w_q + q * C::kHeads;
          const bool fast = allpos && ks > 0.f;
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int hb = 0; hb < 64; hb += 32) {
            float v[32];
            tc::tmem_ld32(taddr + hb, v);
            tc::tmem_ld_wait();
            if (fast) {
#pragma unroll
              for (int h = 0; h < 32; ++h) ps[h & 3] = fmaf(wc[hb + h], fmaxf(v[h], 0.f), ps[h & 3]);
            } else {
#pragma unroll
              for (int h = 0; h < 32; ++h) ps[h & 3] = fmaf(ww[hb + h], fmaxf(v[h] * (wq[hb + h] * ks), 0.f), ps[h & 3]);
            }
          }
          const float sum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
          score[qi] = fast ? sum * ks : sum;
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&acc_empty[acc]);
          tc::mbar_arrive(&sc_empty[r]);
        }
#pragma unroll
        for (int qi = 0; qi < kQPerWarp; ++qi) {
          const int q = NQ == 1 ? 0 : 2 * half + qi;
          const int64_t j = U.j0 + q;
          const bool keep = s < vis_q[qi];
          if (keep) p.scores[(U.b * p.n_q + j) * p.score_stride + s] = score[qi];
          if (do_hist) {
            // lanes with the same bin add their count once (scores crowd into few bins)
            const uint32_t bin = keep ? float_order_key(score[qi]) >> (32 - kTopkHistBits) : 0xFFFFFFFFu;
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (keep && lane == __ffs(peers) - 1)
              atomicAdd(&hist[bin >> 1], (uint32_t)__popc(peers) << (16 * (bin & 1)));
          }
        }
      }
    }
    if (do_hist && ok && hist_row >= 0 && esync()) flush_hist(false);
  }

  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------- host

bool index_tc_shape_supported(const hyb_index_args* a) {
  if (a->dtype != HYB_E4M3 || a->c_I != 128 || a->n_ih != 64) return false;
  const int64_t kvs = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  if (kvs % 4 != 0 || kvs < 1) return false;  // scale rows must start on 16-byte boundaries
  const uintptr_t al = reinterpret_cast<uintptr_t>(a->kI) | reinterpret_cast<uintptr_t>(a->kI_scale) |
                       reinterpret_cast<uintptr_t>(a->qI);
  if (al % 16 != 0) return false;
  if (a->batch * kvs >= (int64_t(1) << 31) || a->batch * a->n_q * 64 >= (int64_t(1) << 31)) return false;
  return true;
}

template <int NQ>
static cudaError_t launch_nq(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                             uint32_t* ghist, bool* hist_done, cudaStream_t s) {
  using C = IdxTc<NQ>;
  const int64_t kvs = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  CUtensorMap tm_keys, tm_scales, tm_q;
  if (!encode_tmap_2d(&tm_keys, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->kI, 128, (uint64_t)(a->batch * kvs), 128, 128,
                      C::kTileE, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a->kI_scale, (uint64_t)kvs, (uint64_t)a->batch,
                      (uint64_t)kvs * 4, C::kTileE, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->qI, 128, (uint64_t)(a->batch * a->n_q * 64), 128, 128,
                      (uint32_t)C::kN, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  IdxTcParams p;
  p.w = a->w, p.qI_scale = a->qI_scale, p.scores = scores, p.score_stride = score_stride;
  p.ghist = nullptr;  // set below once the units are known
  p.n_q = a->n_q, p.n_entries = a->n_entries, p.kv_stride = kvs, p.m = a->m, p.q_pos0 = a->q_pos0;
  p.q_pos = a->q_pos;
  p.groups_per_b = (a->n_q + NQ - 1) / NQ;
  const int64_t groups = p.groups_per_b * a->batch;
  const int64_t tiles_max = (n_vis_max + 127) / 128;
  const int ctas_per_sm = C::kSmemBytes <= 113 * 1024 ? 2 : 1;
  const int64_t slots = (int64_t)kNumSMs * ctas_per_sm;
  // decode: one unit per CTA (one query-group setup, one histogram flush); prefill: two
  // per CTA on average, for balance
  const int64_t per_slot = NQ == 1 ? 1 : 2;
  int64_t tpu = (groups * tiles_max + per_slot * slots - 1) / (per_slot * slots);
  tpu = tpu < 1 ? 1 : (tpu > tiles_max ? tiles_max : tpu);
  p.tiles_per_unit = tpu;
  p.units_per_group = (tiles_max + tpu - 1) / tpu;
  p.n_units = groups * p.units_per_group;
  // fused histogram: one query per unit and fewer than 2^16 entries per unit (16-bit counters)
  if (NQ == 1 && ghist != nullptr && p.tiles_per_unit * C::kTileE < 65536) p.ghist = ghist;
  p.dev_status = a->dev_status;
  if (p.n_units == 0) return cudaSuccess;
  static_assert(NQ != 1 || C::kSmemBytes <= 113 * 1024, "the decode indexer keeps two CTAs per SM");
  cudaError_t e = cudaFuncSetAttribute(index_tc_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.n_units < slots ? p.n_units : slots;
  e = launch_pdl(index_tc_kernel<NQ>, dim3((unsigned)grid), dim3(C::kThreads), (size_t)C::kSmemBytes, s, tm_keys, tm_scales,
                 tm_q, p);
  if (e != cudaSuccess) return e;
  *hist_done = p.ghist != nullptr;
  return cudaGetLastError();
}

cudaError_t launch_index_scores_tc(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                   uint32_t* ghist, bool* hist_done, cudaStream_t s) {
  *hist_done = false;
  if (n_vis_max == 0 || a->n_q == 0 || a->batch == 0) return cudaSuccess;
  if (a->n_q >= 8) return launch_nq<4>(a, scores, score_stride, n_vis_max, nullptr, hist_done, s);
  return launch_nq<1>(a, scores, score_stride, n_vis_max, ghist, hist_done, s);
}

}  // namespace hyb
