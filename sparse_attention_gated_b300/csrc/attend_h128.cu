// attend_h128.cu -- MQA core attention with 128 query heads per CTA on the 5th-generation
// tensor cores (bf16, c = 512, key = value = the compressed entry), for the two compressed
// entry sources of the hybrid-attention forward:
//   mode 0, CSA: the entries listed by the top-k selector ("DeepSeek-V4 hybrid attention"
//           (trishampatil.com) section V.3: every query head attends the same selected
//           entries, key = value = the entry);
//   mode 1, HCA: every visible entry, s < floor((t+1)/m') (same page, section VI);
// each optionally with the query's sliding window fused into the same softmax ("DeepSeek-V4:
// Anatomy..." (modernaiengineering.com), "One query in a CSA layer", steps 4-5: one softmax
// over the union of entries and window rows): as one more split of a decode-shaped launch,
// or as the tiles that follow the list's in a launch with one split.
//
// One CTA owns (query, 128 heads, one half of the 512 output dims, split of the list).
// With the heads on the MMA's 128 rows:
//   S[h,e]  = sum_d Q[h,d] K[e,d]          M = 128 heads, N = 64 entries, K = 512
//   O[h,d] += sum_e P[h,e] V[e,d]          M = 128 heads, N = 256 dims (this half), K = 64
// Tensor memory (512 columns): O (256), Q dims 0..255 as the A operand of S (128 columns
// of bf16 pairs), two S buffers of 64 columns; the softmax writes P (bf16 pairs) over the
// first 32 columns of its S buffer, where the O product reads it as its A operand.  Q dims
// 256..511 stay in shared memory (64 KiB, the A operand of the other half of S).  Both
// halves of a query compute the same S: that buys a whole head group per CTA, so each
// entry is loaded by two CTAs (instead of four loads with 64-head CTAs that each read K
// and V), and each load serves both products (key = value).
// A tile of 64 entries is 8 slabs of [64 rows x 64 dims] bf16 in the 128-byte swizzle.
// The 4 slabs of this CTA's output half go to ring A (freed once O of the tile is done),
// the other 4 to ring B (freed once S is done), so that the next tiles' loads start early.
// Whole tiles of consecutive rows come by TMA tile loads; a ragged last tile and short
// windows by TMA gather4 (a row past the list reads as zeros); index lists by 16-byte
// cp.async copies of two warps, one per ring, written in the swizzled layout (a TMA gather
// moves 4 rows of 128 bytes per instruction, several times slower than the L2 can deliver
// a tile of 64 scattered rows).
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      producer: one lane issues the TMA loads (the query rows; the tiles of
//               contiguous sources), the lanes compute the rows of gather4 copies;
//   warp 1      TMEM owner and MMA issuer (one elected lane);
//   warps 2-3, 8-9  in a CTA with an index list, every tile (the list's, then a fused
//               window's) by cp.async: the other half's slabs (2: rows 0-31, 8: rows 32-63)
//               and this half's (3, 9); warps 2-3 also take part in the split join;
//   warps 4-7   softmax and epilogue: thread h of the four owns TMEM lane h = head h, so a
//               head's scores are one row and its maximum, exponentials and sum stay in
//               one thread.
// Online softmax in base 2 with a lazy reference per head: it moves only when a tile's
// maximum exceeds it by more than 2^8 (then that head's O row is rescaled in TMEM).
// Decode-shaped launches (few queries) split each (query, half) over several CTAs: the splits
// write an unnormalised bf16 partial and (m, l) per head and join through L2 inside the
// kernel (a launch with splits has at most one CTA per SM, so all are resident); each split
// then merges 1/S of the outputs.  Launches with many queries (prefill) run one CTA per
// (query, head group, half) over the whole list and window, with no join.  Every wait is bounded:
// on expiry HYB_DEV_TIMEOUT is raised, the CTA's own copies and products in flight land,
// TMEM is freed and the kernel returns.
#include <cstdlib>

#include "kernels.cuh"
#include "tc_common.cuh"

namespace hyb {

namespace {

constexpr int kH = 128;           // query heads per CTA (MMA M)
constexpr int kC = 512;           // head dim c
constexpr int kT = 64;            // entries per tile (N of the score product)
constexpr int kSlab = kT * 128;   // 8 KiB: [64 rows][64 dims] bf16
constexpr int kQSlab = kH * 128;  // 16 KiB: [128 heads][64 dims] bf16
constexpr int kDA = 3, kDB = 2;   // ring depths in tiles: this CTA's output half / the other half
constexpr int kMaxSplits = 32;  // (the join stages every split's partial slice in the free ring memory)
constexpr int kMaxJoinUnits = kNumSMs / 2;  // arrival and departure words fit the 1 KiB join region
constexpr int kOffQ = 0;
constexpr int kOffA = kOffQ + 4 * kQSlab;
constexpr int kOffB = kOffA + kDA * 4 * kSlab;
constexpr int kOffBar = kOffB + kDB * 4 * kSlab;
enum {
  kBarQ = 0,
  kBarFullA = 1,
  kBarEmptyA = kBarFullA + kDA,
  kBarFullB = kBarEmptyA + kDA,
  kBarEmptyB = kBarFullB + kDB,
  kBarSFull = kBarEmptyB + kDB,
  kBarPFull = kBarSFull + 2,
  kBarODone = kBarPFull + 2,
  kBarQlo = kBarODone + 1,
  kBarFin = kBarQlo + 1,
  kNumBars = kBarFin + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + abort flag, TMEM address; + alignment slack
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;
constexpr int kThreads = 320;
constexpr int kSoftWarp0 = 4;
constexpr int kWarps8 = 8;  // warps 8-9: the second pair of copy warps
constexpr float kTau = 8.0f;          // lazy-reference threshold (log2 units)
constexpr int kOcts = kC / 2 / 8;     // 32 groups of 8 output dims per half

static_assert(kSmemBytes <= 232448, "shared memory budget");

struct H128Params {
  const int32_t* idx;  // mode 0: [rows][list_len]
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;  // the entries [batch][kv_stride][c] (key = value)
  const __nv_bfloat16* wkv; // the window rows [batch][w_stride][c]
  float* o;            // no window: [rows][n_h][c] float32
  float* lse;          // [rows][n_h]: the list's lse, or the union's with a window
  void* out;           // with a window: merged output [rows][n_h][c]
  int out_bf16;
  __nv_bfloat16* part_o;  // splits: [units][n_split][kOcts][128 heads][8 dims]
  float2* part_ml;        // splits: [units][n_split][128 heads] (m in log2 units, l)
  uint32_t* join_cnt;     // splits: [2][kMaxJoinUnits] arrivals and departures (start and end at zero)
  int64_t n_q, n_h, n_entries, kv_stride, list_len, m, q_pos0;
  const int64_t* q_pos;
  int n_split, n_hg, win;
  int64_t w_stride, w_pos0, wq_pos0, n_win;
  const int64_t* wq_pos;
  const int64_t* w_pos0s;
  int32_t k_rows, w_rows;  // row counts of the entry and window tensor maps (a row index there reads zeros)
  float scale_log2;
  int32_t* dev_status;
  long long wait_cycles;
  const float* sink;  // optional per-head sink logits [n_h] (natural log), joined to the final result
};

struct H128Work {
  int64_t bq, b, j, hg, dh, sp, unit;
  int64_t L;     // list length of this split's source
  int64_t row0;  // contiguous sources: map row of list position 0
  const int32_t* list;
  int64_t tb, te;  // this split's tiles
  bool win;        // the split attends the window (contiguous rows of the window map)
  // one split with a window: the window's tiles follow the list's (rows wrow0 .. wrow0 + wL - 1)
  int64_t nw, wL, wrow0;
};

// 2^x by the SFU's approximate exponential (relative error far below the bf16 rounding
// the probabilities get next; 2^-inf = 0).
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The final normaliser of a head whose softmax has base-2 maximum m and sum l (l = 0: no
// entry), with the head's sink logit s (natural log; -inf = none) as one more term of the
// denominator with no value: returns the factor that replaces 1 / l on the accumulated
// output and writes the union's natural-log lse (no entry: output 0, lse = s).
__device__ __forceinline__ float sink_normaliser(float m, float l, float s, float& lse) {
  if (!(l > 0.f)) {
    lse = s;
    return 0.f;
  }
  const float s2 = s * kLog2e;
  const float M = fmaxf(m, s2);
  const float a = ex2_sfu(m - M), den = fmaf(l, a, ex2_sfu(s2 - M));
  lse = (M + __log2f(den)) * kLn2;
  return a / den;
}

template <int MODE>
__device__ __forceinline__ H128Work h128_work(const H128Params& p) {
  H128Work w;
  const int64_t id = blockIdx.x;  // split fastest: the splits of a unit are consecutive CTAs
  w.sp = id % p.n_split;
  w.unit = id / p.n_split;
  w.dh = w.unit & 1;
  w.hg = (w.unit >> 1) % p.n_hg;
  w.bq = (w.unit >> 1) / p.n_hg;
  w.b = w.bq / p.n_q;
  w.j = w.bq % p.n_q;
  const bool report = w.hg == 0 && w.dh == 0 && threadIdx.x == 0;
  w.list = nullptr;
  w.row0 = 0;
  w.win = false;
  w.nw = 0, w.wL = 0, w.wrow0 = 0;
  if (p.win && p.n_split > 1 && w.sp == p.n_split - 1) {
    const int64_t tw = query_pos(p.wq_pos, p.wq_pos0, w.bq, w.j);
    const int64_t kvp = p.w_pos0s ? __ldg(p.w_pos0s + w.b) : p.w_pos0;
    int64_t first;
    w.win = true;
    w.L = window_rows(tw, p.n_win, kvp, p.w_stride, &first, p.dev_status, report);
    w.row0 = w.b * p.w_stride + first;
    w.tb = 0;
    w.te = (w.L + kT - 1) / kT;
    return w;
  }
  if constexpr (MODE == 0) {
    w.L = p.list_len;
    w.list = p.idx + w.bq * p.list_len;
  } else {
    const int64_t t = query_pos(p.q_pos, p.q_pos0, w.bq, w.j);
    w.L = visible_checked(t, p.m, p.n_entries, p.dev_status, report && w.sp == 0);
    w.row0 = w.b * p.kv_stride;
  }
  const int64_t T = (w.L + kT - 1) / kT;
  const int64_t S = p.n_split - (p.win && p.n_split > 1 ? 1 : 0);
  w.tb = w.sp * T / S;
  w.te = (w.sp + 1) * T / S;
  if (p.win && p.n_split == 1) {
    const int64_t tw = query_pos(p.wq_pos, p.wq_pos0, w.bq, w.j);
    const int64_t kvp = p.w_pos0s ? __ldg(p.w_pos0s + w.b) : p.w_pos0;
    int64_t first;
    w.wL = window_rows(tw, p.n_win, kvp, p.w_stride, &first, p.dev_status, report);
    w.wrow0 = w.b * p.w_stride + first;
    w.nw = (w.wL + kT - 1) / kT;
  }
  return w;
}

// Map row of list position pos, or `oob` (a row index that reads zeros) when the position
// holds no entry.  report: flag an index outside [-1, n_entries).
template <int MODE>
__device__ __forceinline__ int32_t h128_row(const H128Params& p, const H128Work& w, int64_t pos, int32_t oob,
                                            bool report) {
  if (pos >= w.L) return oob;
  if (MODE == 0 && !w.win) {
    const int32_t s = __ldg(w.list + pos);
    if (s < 0 || s >= p.n_entries) {
      if (report && s != -1) flag_status(p.dev_status, HYB_DEV_BAD_INDEX);
      return oob;
    }
    return (int32_t)(w.b * p.kv_stride + s);
  }
  return (int32_t)(w.row0 + pos);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attend_h128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_kg, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_wg, H128Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + kOffQ;
  uint8_t* ring_a = smem + kOffA;
  uint8_t* ring_b = smem + kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + kBarQ;
  uint64_t* full_a = bars + kBarFullA;
  uint64_t* empty_a = bars + kBarEmptyA;
  uint64_t* full_b = bars + kBarFullB;
  uint64_t* empty_b = bars + kBarEmptyB;
  uint64_t* s_full = bars + kBarSFull;
  uint64_t* p_full = bars + kBarPFull;
  uint64_t* o_done = bars + kBarODone;
  uint64_t* qlo_ready = bars + kBarQlo;
  uint64_t* fin = bars + kBarFin;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // positions in device memory may have been written by the previous kernel: read them after the wait
  if (p.q_pos != nullptr || p.wq_pos != nullptr || p.w_pos0s != nullptr) pdl_wait();
  const H128Work W = h128_work<MODE>(p);
  const int64_t nl = W.te - W.tb;  // tiles of the list (or of the window split's window)
  const int64_t ntiles = nl + W.nw;  // + the window's, after them, with one split
  const bool contig = MODE != 0 || W.win;
  // index-list tiles are copied by warps 2-3, and then every tile of the CTA is (so that one
  // role fills the rings in tile order: a parity wait on a slot's barrier is only exact for
  // the next phase)
  const bool gathered = !contig;

  if (threadIdx.x == 0) {
    // a tile's slabs in a ring: one TMA transaction count, or two copy warps' signals
    const uint32_t nfull = gathered ? 2 : 1;
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < kDA; ++s) tc::mbar_init(&full_a[s], nfull), tc::mbar_init(&empty_a[s], 1);
    for (int s = 0; s < kDB; ++s) tc::mbar_init(&full_b[s], nfull), tc::mbar_init(&empty_b[s], 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&s_full[i], 1), tc::mbar_init(&p_full[i], 4);
    tc::mbar_init(o_done, 1);
    tc::mbar_init(qlo_ready, 4);
    tc::mbar_init(fin, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(s_tmem, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // (before it: shared memory, TMEM and parameters only)
  pdl_trigger();

  const int64_t qrow = W.bq * p.n_h + W.hg * kH;  // first head row of this CTA in q / o / out
  if (warp == 0) {
    // ================================================================ producer
    bool ok = true;
    int64_t last_a[kDA], last_b[kDB];  // last tile issued into each slot (drained on abort)
#pragma unroll
    for (int s = 0; s < kDA; ++s) last_a[s] = -1;
#pragma unroll
    for (int s = 0; s < kDB; ++s) last_b[s] = -1;
    const CUtensorMap* tmt_l = W.win ? &tm_w : &tm_k;
    const CUtensorMap* tmg_l = W.win ? &tm_wg : &tm_kg;
    const int32_t oob_l = W.win ? p.w_rows : p.k_rows;
    // the query rows: dims 256..511 into their own region, dims 0..255 staged in ring A's
    // slots 1 and 2 until the softmax warps have moved them into TMEM
    if (ntiles > 0 && lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::mbar_arrive_expect_tx(q_full, 8 * kQSlab);
      for (int s = 0; s < 4; ++s) {
        tc::tma_load_2d(q_s + s * kQSlab, &tm_q, q_full, 256 + 64 * s, (int32_t)qrow);
        tc::tma_load_2d(ring_a + 4 * kSlab + s * kQSlab, &tm_q, q_full, 64 * s, (int32_t)qrow);
      }
      tc::prefetch_tmap(tmt_l);
      tc::prefetch_tmap(tmg_l);
      if (W.nw > 0) tc::prefetch_tmap(&tm_w), tc::prefetch_tmap(&tm_wg);
    }
    bool qlo_seen = false;
    for (int64_t li = 0; li < (gathered ? 0 : ntiles) && ok; ++li) {
      const bool wt = li >= nl;  // a window tile after the list's
      const int64_t i = wt ? li - nl : W.tb + li;
      const CUtensorMap* tmt = wt ? &tm_w : tmt_l;
      const CUtensorMap* tmg = wt ? &tm_wg : tmg_l;
      const int32_t oob = wt ? p.w_rows : oob_l;
      if (li >= 1 && !qlo_seen) {
        // ring A's slots 1 and 2 hold the staged query rows until they are in TMEM
        int okq = 1;
        if (lane == 0) okq = tc::mbar_wait(qlo_ready, 0, s_abort, 12);
        if (!(ok = __shfl_sync(0xffffffffu, okq, 0) != 0)) break;
        qlo_seen = true;
      }
      const int sa = (int)(li % kDA), sb = (int)(li % kDB);
      const bool whole = wt ? (i + 1) * kT <= W.wL : contig && (i + 1) * kT <= W.L;
      int32_t r0 = oob, r1 = oob;  // map rows of positions 64i + lane and 64i + 32 + lane
      if (!whole && wt) {
        const int64_t p0 = i * kT + lane, p1 = p0 + 32;
        r0 = p0 < W.wL ? (int32_t)(W.wrow0 + p0) : oob;
        r1 = p1 < W.wL ? (int32_t)(W.wrow0 + p1) : oob;
      } else if (!whole) {
        r0 = h128_row<MODE>(p, W, i * kT + lane, oob, true);
        r1 = h128_row<MODE>(p, W, i * kT + 32 + lane, oob, true);
      }
      int okl = 1;
      if (lane == 0) {
        okl = tc::mbar_wait(&empty_b[sb], (uint32_t)((li / kDB) & 1) ^ 1u, s_abort, 1) &&
              tc::mbar_wait(&empty_a[sa], (uint32_t)((li / kDA) & 1) ^ 1u, s_abort, 2);
        if (okl) {
          tc::mbar_arrive_expect_tx(&full_b[sb], 4 * kSlab);
          tc::mbar_arrive_expect_tx(&full_a[sa], 4 * kSlab);
          last_a[sa] = li, last_b[sb] = li;
        }
      }
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      if (!ok) break;
      if (whole) {
        if (lane == 0) {
          const int32_t y = (int32_t)((wt ? W.wrow0 : W.row0) + i * kT);
          for (int j = 0; j < 4; ++j) {
            const int own = 4 * (int)W.dh + j, other = 4 * (1 - (int)W.dh) + j;
            tc::tma_load_2d(ring_b + (sb * 4 + j) * kSlab, tmt, &full_b[sb], 64 * other, y);
            tc::tma_load_2d(ring_a + (sa * 4 + j) * kSlab, tmt, &full_a[sa], 64 * own, y);
          }
        }
      } else {
        // lane g < 16 gathers rows 4g .. 4g+3 of the tile into every slab
        int32_t y[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int srcl = (4 * lane + q) & 31;
          const int32_t a0 = __shfl_sync(0xffffffffu, r0, srcl);
          const int32_t a1 = __shfl_sync(0xffffffffu, r1, srcl);
          y[q] = lane < 8 ? a0 : a1;
        }
        if (lane < 16) {
          for (int j = 0; j < 4; ++j) {
            const int own = 4 * (int)W.dh + j, other = 4 * (1 - (int)W.dh) + j;
            tc::tma_gather4(ring_b + (sb * 4 + j) * kSlab + lane * 512, tmg, &full_b[sb], 64 * other, y[0], y[1],
                            y[2], y[3]);
            tc::tma_gather4(ring_a + (sa * 4 + j) * kSlab + lane * 512, tmg, &full_a[sa], 64 * own, y[0], y[1], y[2],
                            y[3]);
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // let this thread's copies in flight land before the CTA can exit
      for (int s = 0; s < kDA; ++s)
        if (last_a[s] >= 0) tc::mbar_wait_drain(&full_a[s], (uint32_t)((last_a[s] / kDA) & 1));
      for (int s = 0; s < kDB; ++s)
        if (last_b[s] >= 0) tc::mbar_wait_drain(&full_b[s], (uint32_t)((last_b[s] / kDB) & 1));
      if (ntiles > 0) tc::mbar_wait_drain(q_full, 0);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (tc::elect_one()) {
      bool ok = ntiles == 0 || (tc::mbar_wait(q_full, 0, s_abort, 3) && tc::mbar_wait(qlo_ready, 0, s_abort, 4));
      constexpr uint32_t idS = tc::make_idesc(1, 1, 0, 0, kH, kT);   // A = Q (K-major), B = K rows (K-major)
      constexpr uint32_t idO = tc::make_idesc(1, 1, 0, 1, kH, 256);  // A = P (TMEM), B = V rows (MN-major)
      const uint32_t q_addr = tc::smem_u32(q_s), a_addr = tc::smem_u32(ring_a), b_addr = tc::smem_u32(ring_b);
      // S of tile li in two parts: the other half's slabs (ring B, whose slot is freed as
      // soon as they are consumed), then this half's (ring A, freed after O of the tile)
      auto issue_s_part = [&](int64_t li, int part) {
        const int b = (int)(li & 1), sa = (int)(li % kDA), sb = (int)(li % kDB);
        const bool other = part == 0;
        const uint32_t dS = tmem + kColS + 64u * b;
        tc::tc_fence_after();
        for (int j = 0; j < 4; ++j) {
          const int slab = other ? 4 * (1 - (int)W.dh) + j : 4 * (int)W.dh + j;  // dims 64*slab ..
          const uint32_t kslab =
              other ? b_addr + (uint32_t)((sb * 4 + j) * kSlab) : a_addr + (uint32_t)((sa * 4 + j) * kSlab);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = tc::desc_kmajor_sw128(kslab + 32 * kk);
            const uint32_t acc = (part == 1 || j > 0 || kk > 0) ? 1u : 0u;
            if (slab < 4)  // Q dims 0..255 from TMEM: bf16 pairs, 8 columns per 16 dims
              tc::mma_f16_ts(dS, tmem + kColQ + (uint32_t)(32 * slab + 8 * kk), bd, idS, acc);
            else
              tc::mma_f16(dS, tc::desc_kmajor_sw128(q_addr + (slab - 4) * kQSlab + 32 * kk), bd, idS, acc);
          }
        }
        if (other)
          tc::mma_commit(&empty_b[sb]);
        else
          tc::mma_commit(&s_full[b]);
      };
      auto issue_o = [&](int64_t li) {
        const int b = (int)(li & 1), sa = (int)(li % kDA);
        tc::tc_fence_after();
        const uint32_t v0 = a_addr + (uint32_t)(sa * 4 * kSlab);
#pragma unroll
        for (int ks = 0; ks < kT / 16; ++ks)
          tc::mma_f16_ts(tmem + kColO, tmem + kColS + 64u * b + 8u * ks,
                         tc::desc_mnmajor_sw128(v0 + ks * 2048, kSlab, 1024), idO, (li > 0 || ks > 0) ? 1u : 0u);
        tc::mma_commit(&empty_a[sa]);
        tc::mma_commit(o_done);
      };
      // Issue whatever is ready, O first: O of tile no as soon as its probabilities are
      // written, S of tile ns (part by part) as soon as its slabs are in and its S buffer
      // is free (O of tile ns-2 issued).  A late tile then never holds back the O product
      // that frees an earlier tile's slot.  Bounded like every wait.
      int64_t ns = 0, no = 0;
      int spart = 0;
      long long t0 = clock64();
      uint32_t spins = 0;
      while (ok && no < ntiles) {
        bool progress = false;
        if (no < ns && tc::mbar_try_wait(&p_full[no & 1], (uint32_t)((no >> 1) & 1))) {
          issue_o(no++);
          progress = true;
        } else if (ns < ntiles && ns <= no + 1) {
          if (spart == 0 && tc::mbar_try_wait(&full_b[ns % kDB], (uint32_t)((ns / kDB) & 1))) {
            issue_s_part(ns, 0);
            spart = 1;
            progress = true;
          } else if (spart == 1 && tc::mbar_try_wait(&full_a[ns % kDA], (uint32_t)((ns / kDA) & 1))) {
            issue_s_part(ns++, 1);
            spart = 0;
            progress = true;
          }
        }
        if (progress) {
          t0 = clock64();
          spins = 0;
        } else if ((++spins & 15) == 0) {
          if (*s_abort) {
            ok = false;
          } else if (clock64() - t0 > tc::kWaitLimitCycles) {
            *s_abort = 5;
            ok = false;
          }
        }
      }
      // every MMA issued above has completed once `fin` flips
      tc::mma_commit(fin);
      tc::mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else if (gathered && (warp == 2 || warp == 3 || warp >= kWarps8)) {
    // ================================================================ tiles by cp.async
    // Warps 2 and 8 copy the other half's 4 slabs of each tile (the list's, then the
    // window's) into ring B, warps 3 and 9 this half's into ring A; warps 2-3 take the
    // tile's rows 0-31, warps 8-9 rows 32-63 (a warp issues one 512-byte cp.async in some 30
    // cycles, so a tile needs four warps to keep up with the L2).  Lane l copies 16-byte
    // chunk l % 8 of rows 4u + l / 8 of the warp's 32 rows in every slab: one instruction
    // moves four 128-byte row pieces.  A tile's copies are one group; the warp signals the
    // tile's full barrier (two signals complete it) once the group has landed (checked
    // while the next tile's copies are in flight), after a proxy fence that hands the writes
    // to the tensor cores.  Positions without an entry are written as zeros.
    const bool own = (warp & 1) != 0;
    const int part = warp >= kWarps8 ? 1 : 0;  // rows 32 part .. 32 part + 31
    const int c16 = lane & 7;
    const int half = own ? (int)W.dh : 1 - (int)W.dh;
    const char* kbase = reinterpret_cast<const char*>(p.kv);
    const char* wbase = reinterpret_cast<const char*>(p.wkv);
    uint8_t* ring = own ? ring_a : ring_b;
    const int depth = own ? kDA : kDB;
    int32_t nx0 = -1, nx1 = -1;  // list values at positions lane and 32 + lane of the next tile
    auto fetch = [&](int64_t li_) {
      const int64_t pos = (W.tb + li_) * kT + lane;
      nx0 = pos < W.L ? __ldg(W.list + pos) : -1;
      nx1 = pos + 32 < W.L ? __ldg(W.list + pos + 32) : -1;
    };
    // map row of a list value; -1 when it holds no entry (an index outside [-1, n_entries)
    // is reported and left out)
    auto map_row = [&](int32_t v, bool report) -> int32_t {
      if (v < 0 || v >= p.n_entries) {
        if (v != -1 && report) flag_status(p.dev_status, HYB_DEV_BAD_INDEX);
        return -1;
      }
      return (int32_t)(W.b * p.kv_stride + v);
    };
    auto signal = [&](int64_t lt) {
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(own ? &full_a[lt % kDA] : &full_b[lt % kDB]);
    };
    if (nl > 0) fetch(0);
    int64_t pend = -1;  // the tile whose copies are in flight and not yet signalled
    bool ok = true;
    for (int64_t li = 0; li < ntiles && ok; ++li) {
      const bool wt = li >= nl;  // a window tile (rows wrow0 + position)
      int32_t mr_l;  // map row of position 32 part + lane of the tile (-1: none)
      if (wt) {
        const int64_t pw = (li - nl) * kT + 32 * part + lane;
        mr_l = pw < W.wL ? (int32_t)(W.wrow0 + pw) : -1;
      } else {
        mr_l = map_row(part ? nx1 : nx0, !own);
        if (li + 1 < nl) fetch(li + 1);
      }
      const char* base = wt ? wbase : kbase;
      int32_t rows[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) rows[u] = __shfl_sync(0xffffffffu, mr_l, 4 * u + (lane >> 3));
      const int slot = (int)(li % depth);
      int okw = 1;
      if (lane == 0) {
        okw = tc::mbar_wait(own ? &empty_a[slot] : &empty_b[slot], (uint32_t)((li / depth) & 1) ^ 1u, s_abort, 20);
        // ring A's slots 1 and 2 hold the staged query rows until they are in TMEM
        if (okw && own && li == 1) okw = tc::mbar_wait(qlo_ready, 0, s_abort, 21);
      }
      if (!(ok = __shfl_sync(0xffffffffu, okw, 0) != 0)) break;
      const uint32_t dst0 = tc::smem_u32(ring + slot * 4 * kSlab);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int sd = 4 * half + j;  // the slab's 64 dims of the row
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = 32 * part + 4 * u + (lane >> 3);
          const int32_t mr = rows[u];
          const char* src = base + (int64_t)(mr < 0 ? 0 : mr) * (kC * 2) + sd * 128 + c16 * 16;
          tc::cp_async16(dst0 + (uint32_t)(j * kSlab + r * 128 + ((c16 ^ (r & 7)) << 4)), src, mr < 0 ? 0u : 16u);
        }
      }
      tc::cp_async_commit();
      if (pend >= 0) {
        tc::cp_async_wait_group<1>();
        signal(pend);
      }
      pend = li;
    }
    tc::cp_async_wait_group<0>();  // (after an abort too: the copies land before the CTA exits)
    if (ok && pend >= 0) signal(pend);
  } else if (warp >= kSoftWarp0 && warp < kWarps8) {
    // ================================================================ softmax + epilogue
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;  // head (TMEM lane) of this thread
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    bool ok = true;
    if (ntiles > 0) {
      // Q dims 0..255 of head h (staged by TMA in ring A, 128-byte swizzle: 16-byte chunk c
      // of row h at chunk c ^ (h & 7)) into TMEM, the A operand of S: 128 columns of bf16 pairs
      ok = tc::mbar_wait(q_full, 0, s_abort, 13);
      if (ok) {
        const uint8_t* stage = ring_a + 4 * kSlab + h * 128;
#pragma unroll 1
        for (int sl = 0; sl < 4; ++sl) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(stage + sl * kQSlab + ((c ^ (h & 7)) << 4));
            v[4 * c] = u.x, v[4 * c + 1] = u.y, v[4 * c + 2] = u.z, v[4 * c + 3] = u.w;
          }
          tc::tmem_st32u(tmem + lane_base + kColQ + 32u * sl, v);
        }
        tc::tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(qlo_ready);
      }
    }
    float m = -INFINITY, l = 0.f;  // reference (log2 units) and denominator of head h
    // list values of the next list tile at positions lane and 32 + lane (loaded a tile ahead)
    int32_t nx0 = -1, nx1 = -1;
    auto fetch = [&](int64_t li_) {
      const int64_t pos = (W.tb + li_) * kT + lane;
      nx0 = pos < W.L ? __ldg(W.list + pos) : -1;
      nx1 = pos + 32 < W.L ? __ldg(W.list + pos + 32) : -1;
    };
    if (gathered && nl > 0) fetch(0);
    for (int64_t li = 0; li < ntiles && ok; ++li) {
      const bool wt = li >= nl;
      const int64_t i = wt ? li - nl : W.tb + li;
      const int b = (int)(li & 1);
      // which of the tile's 64 entries exist
      uint64_t valid;
      if (wt || contig) {
        const int64_t n = (wt ? W.wL : W.L) - i * kT;
        valid = n >= kT ? ~0ull : ((1ull << n) - 1ull);
      } else {
        const bool v0 = nx0 >= 0 && nx0 < p.n_entries, v1 = nx1 >= 0 && nx1 < p.n_entries;
        if (li + 1 < nl) fetch(li + 1);
        valid = (uint64_t)__ballot_sync(0xffffffffu, v0) | ((uint64_t)__ballot_sync(0xffffffffu, v1) << 32);
      }
      if (!(ok = tc::mbar_wait(&s_full[b], (uint32_t)((li >> 1) & 1), s_abort, 8))) break;
      tc::tc_fence_after();
      float s[64];
      {
        float t0[32], t1[32];
        tc::tmem_ld32(tmem + lane_base + kColS + 64u * b, t0);
        tc::tmem_ld32(tmem + lane_base + kColS + 64u * b + 32u, t1);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = t0[e], s[32 + e] = t1[e];
      }
      if (valid == ~0ull) {
#pragma unroll
        for (int e = 0; e < 64; ++e) s[e] *= p.scale_log2;
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) s[e] = ((valid >> e) & 1ull) ? s[e] * p.scale_log2 : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) mx[x] = s[x];
#pragma unroll
      for (int e = 8; e < 64; ++e) mx[e & 7] = fmaxf(mx[e & 7], s[e]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // lazy reference: moves only when the tile's maximum exceeds it by more than 2^kTau
      const bool mv = mt > m + kTau || (m == -INFINITY && mt != -INFINITY);
      float alpha = 1.f;
      if (mv) {
        alpha = m == -INFINITY ? 0.f : exp2f(m - mt);
        m = mt;
        l *= alpha;
      }
      if (__any_sync(0xffffffffu, mv && li > 0)) {
        // rescale this head's O row once the previous tile's product is done
        if (!(ok = tc::mbar_wait(o_done, (uint32_t)((li - 1) & 1), s_abort, 9))) break;
        tc::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float v[32];
          tc::tmem_ld32(tmem + lane_base + kColO + 32u * c, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] *= alpha;
          tc::tmem_st32(tmem + lane_base + kColO + 32u * c, v);
        }
        tc::tmem_st_wait();
      }
      // probabilities of head h over the tile (bf16 pairs over the first 32 S columns)
      uint32_t pk[32];
      float ls[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) ls[x] = 0.f;
      const float mref = m != -INFINITY ? m : 0.f;  // (every score is -inf while there is no reference)
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const float p0 = ex2_sfu(s[2 * x] - mref);
        const float p1 = ex2_sfu(s[2 * x + 1] - mref);
        ls[x & 7] += p0 + p1;
        pk[x] = pack_bf16x2(p0, p1);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tc::tmem_st32u(tmem + lane_base + kColS + 64u * b, pk);
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&p_full[b]);
    }
    // ---------------------------------------------------------------- epilogue
    // every product done: `fin` completes once, after the last one (a parity wait on o_done,
    // which completes once per tile, could pass on an earlier phase)
    if (ok && ntiles > 0) {
      ok = tc::mbar_wait(fin, 0, s_abort, 10);
      tc::tc_fence_after();
    }
    if (ok && p.n_split > 1) {
      // split partial: (m, l) of head h; its O row is written below by all eight warps
      p.part_ml[(W.unit * p.n_split + W.sp) * kH + h] = make_float2(l > 0.f ? m : -INFINITY, l);
    } else if (ok) {
      // one split: the normalised output of this half (float32 o, or with a window the
      // merged out in its own type) and the lse
      float lse_h = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
      const float inv = p.sink ? sink_normaliser(m, l, p.sink[W.hg * kH + h], lse_h) : (l > 0.f ? 1.f / l : 0.f);
      const int64_t at = (qrow + h) * kC + 256 * W.dh;
      const bool to_bf16 = p.win && p.out_bf16;
      float* dst = p.win ? static_cast<float*>(p.out) + at : p.o + at;
      __nv_bfloat16* dst16 = static_cast<__nv_bfloat16*>(p.out) + at;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float v[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tmem + lane_base + kColO + 32u * c, v);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] = 0.f;
        }
        if (to_bf16) {
#pragma unroll
          for (int x = 0; x < 4; ++x)
            *reinterpret_cast<uint4*>(dst16 + 32 * c + 8 * x) =
                make_uint4(pack_bf16x2(v[8 * x] * inv, v[8 * x + 1] * inv), pack_bf16x2(v[8 * x + 2] * inv, v[8 * x + 3] * inv),
                           pack_bf16x2(v[8 * x + 4] * inv, v[8 * x + 5] * inv), pack_bf16x2(v[8 * x + 6] * inv, v[8 * x + 7] * inv));
        } else {
#pragma unroll
          for (int x = 0; x < 8; ++x)
            *reinterpret_cast<float4*>(dst + 32 * c + 4 * x) =
                make_float4(v[4 * x] * inv, v[4 * x + 1] * inv, v[4 * x + 2] * inv, v[4 * x + 3] * inv);
        }
      }
      if (W.dh == 0) p.lse[qrow + h] = lse_h;
    }
    if (!ok && *s_abort == 0) *s_abort = 11;
  }

  // ==================================================================== split join
  __syncwarp();
  if (p.n_split > 1) {
    // this split's unnormalised O, bf16, [oct][head][8 dims]: warp w reads TMEM lane quadrant
    // w % 4 (heads 32(w%4) ..) and columns 128 (w / 4) .. 128 (w / 4) + 127
    if (ntiles > 0 && *s_abort == 0 && warp < kWarps8) {
      bool fine = tc::mbar_wait(fin, 0, s_abort, 10);
      if (fine) {
        tc::tc_fence_after();
        const int q4 = warp & 3, hh = q4 * 32 + lane, c0 = (warp >> 2) * 4;  // (warps 0-7)
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        __nv_bfloat16* dst = p.part_o + (W.unit * p.n_split + W.sp) * (int64_t)(kOcts * kH * 8);
        float v[2][32];
        tc::tmem_ld32(tmem + lane_base + kColO + 32u * c0, v[0]);
        tc::tmem_ld32(tmem + lane_base + kColO + 32u * (c0 + 1), v[1]);
        tc::tmem_ld_wait();
#pragma unroll 1
        for (int cc = 0; cc < 4; cc += 2) {
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int oct = 4 * (c0 + cc + u) + x;
              *reinterpret_cast<uint4*>(dst + ((int64_t)oct * kH + hh) * 8) =
                  make_uint4(pack_bf16x2(v[u][8 * x], v[u][8 * x + 1]), pack_bf16x2(v[u][8 * x + 2], v[u][8 * x + 3]),
                             pack_bf16x2(v[u][8 * x + 4], v[u][8 * x + 5]), pack_bf16x2(v[u][8 * x + 6], v[u][8 * x + 7]));
            }
          if (cc == 0) {
            tc::tmem_ld32(tmem + lane_base + kColO + 32u * (c0 + 2), v[0]);
            tc::tmem_ld32(tmem + lane_base + kColO + 32u * (c0 + 3), v[1]);
            tc::tmem_ld_wait();
          }
        }
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort == 0) {
      uint32_t* cnt = p.join_cnt + W.unit;
      uint32_t* dep = p.join_cnt + kMaxJoinUnits + W.unit;
      __threadfence();
      atomicAdd(cnt, 1u);
      const long long t0 = clock64();
      bool joined = true;
      while (tc::ld_acquire_gpu_u32(cnt) < (uint32_t)p.n_split) {
        if (clock64() - t0 > p.wait_cycles) {
          *s_abort = 18;
          joined = false;
          break;
        }
      }
      __threadfence();
      // the last split past the barrier puts both counters back to zero for the next call
      if (joined && atomicAdd(dep, 1u) == (uint32_t)(p.n_split - 1)) {
        atomicExch(cnt, 0u);
        atomicExch(dep, 0u);
      }
    }
    __syncthreads();
    if (*s_abort == 0) {
      // Split sp merges items [i0, i1) of the unit's 32 octs x 128 heads.  The items' partials
      // are consecutive 16-byte pieces in every split's [oct][head][8] block, so one bulk copy
      // per split brings them into the free ring memory, with every split's (m, l) of the 128
      // heads: all in flight at once, one round trip.  The merge then reads shared memory.
      constexpr int kItems = kOcts * kH;
      const int S = p.n_split;
      const int i0 = (int)((int64_t)W.sp * kItems / S), i1 = (int)((int64_t)(W.sp + 1) * kItems / S);
      const int n_it = i1 - i0;
      uint4* st_o = reinterpret_cast<uint4*>(ring_a);                       // [S][n_it]
      float2* st_ml = reinterpret_cast<float2*>(ring_a + S * n_it * 16);  // [S][128]
      if (warp == 0) {
        // lane sp issues split sp's two copies (the transaction count is set first)
        if (lane == 0) tc::mbar_arrive_expect_tx(q_full, (uint32_t)(S * (n_it * 16 + kH * 8)));
        __syncwarp();
        tc::fence_proxy_async_global();  // the other splits' generic writes, acquired above, before these async reads
        const float2* ml_u = p.part_ml + W.unit * (int64_t)S * kH;
        const __nv_bfloat16* po_u = p.part_o + W.unit * (int64_t)S * (kOcts * kH * 8);
        for (int sp = lane; sp < S; sp += 32) {
          tc::bulk_load(st_o + sp * n_it, po_u + ((int64_t)sp * kItems + i0) * 8, (uint32_t)(n_it * 16), q_full);
          tc::bulk_load(st_ml + sp * kH, ml_u + (int64_t)sp * kH, kH * 8, q_full);
        }
      }
      // (q_full completed its first phase when the query rows landed, or never if this split
      // had no tile: wait for the phase after that one)
      const bool staged = tc::mbar_wait(q_full, ntiles > 0 ? 1u : 0u, s_abort, 19);
      for (int it = i0 + (int)threadIdx.x; staged && it < i1; it += kThreads) {
        const int oct = it / kH, hh = it - oct * kH, k = it - i0;
        float M = -INFINITY;
#pragma unroll 4
        for (int sp = 0; sp < S; ++sp) M = fmaxf(M, st_ml[sp * kH + hh].x);
        float L = 0.f, acc[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[x] = 0.f;
        if (M != -INFINITY) {
#pragma unroll 4
          for (int sp = 0; sp < S; ++sp) {
            const float2 ml = st_ml[sp * kH + hh];
            if (ml.x == -INFINITY) continue;
            const float e = ex2_sfu(ml.x - M);
            L = fmaf(ml.y, e, L);
            const uint4 raw = st_o[sp * n_it + k];
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[x]));
              acc[2 * x] = fmaf(e, v.x, acc[2 * x]);
              acc[2 * x + 1] = fmaf(e, v.y, acc[2 * x + 1]);
            }
          }
        }
        float lse_h = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        const float inv = p.sink ? sink_normaliser(M, L, p.sink[W.hg * kH + hh], lse_h) : (L > 0.f ? 1.f / L : 0.f);
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[x] *= inv;
        if (W.dh == 0 && oct == 0) p.lse[qrow + hh] = lse_h;
        const int64_t at = (qrow + hh) * kC + 256 * W.dh + 8 * oct;
        if (p.win && p.out_bf16) {
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + at) =
              make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                         pack_bf16x2(acc[6], acc[7]));
        } else {
          float* dst = p.win ? static_cast<float*>(p.out) : p.o;
          *reinterpret_cast<float4*>(dst + at) = make_float4(acc[0], acc[1], acc[2], acc[3]);
          *reinterpret_cast<float4*>(dst + at + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
      }
      if (!staged && threadIdx.x == 0) tc::mbar_wait_drain(q_full, ntiles > 0 ? 1u : 0u);  // let the copies land
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT | ((*s_abort & 0xFF) << 8));
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

int64_t h128_list_len_max(const AttendJob& j) {
  if (j.mode == 0) return j.list_len;
  return j.q_pos ? j.n_entries : std::min<int64_t>(visible_entries(j.q_pos0 + j.n_q - 1, j.m), j.n_entries);
}

struct H128Plan {
  int n_split;
};

// Splits per (query, head group, half): as many as fit one CTA per SM, evened out (the
// same tiles per split, fewer CTAs); a fused window is one more split, the last.  Launches
// with more units than that (every unit at least two CTAs, all resident) have one split.
H128Plan h128_plan(const AttendJob& j) {
  const int64_t units = j.batch * j.n_q * (j.n_h / kH) * 2;
  if (units * 2 > kNumSMs || units > kMaxJoinUnits) return {1};
  const int w = j.win ? 1 : 0;
  const int64_t T = (h128_list_len_max(j) + kT - 1) / kT;
  int64_t s = kNumSMs / std::max<int64_t>(units, 1) - w;
  s = std::min<int64_t>(std::min<int64_t>(s, std::max<int64_t>(T, 1)), kMaxSplits - w);
  if (s < 1) s = 1;
  const int64_t per = (T + s - 1) / s;
  const int64_t used = per > 0 ? (T + per - 1) / per : 1;
  return {(int)(std::max<int64_t>(used, 1) + w)};
}

}  // namespace

// On unless the environment sets HYB_ATTEND_H128=0 (read once): a switch for measuring the
// 64-head kernel on the same shapes.
bool attend_h128_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("HYB_ATTEND_H128");
    return v == nullptr || v[0] != '0';
  }();
  return on;
}

bool attend_h128_supported(const AttendJob& j) {
  if (j.mode != 0 && j.mode != 1) return false;
  if (j.dtype != HYB_BF16 || j.c != kC || j.n_h < kH || j.n_h % kH != 0 || j.k != j.v) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(j.q) | reinterpret_cast<uintptr_t>(j.k);
  if (al % 16 != 0) return false;
  if (j.batch * j.kv_stride >= (int64_t(1) << 31) - 1 || j.batch * j.n_q * j.n_h >= (int64_t(1) << 31)) return false;
  if (j.win) {
    if (reinterpret_cast<uintptr_t>(j.wk) % 16 != 0 || j.batch * j.w_stride >= (int64_t(1) << 31) - 1) return false;
  }
  return true;
}

int attend_h128_splits(const AttendJob& j) { return h128_plan(j).n_split; }

size_t attend_h128_workspace_bytes(const AttendJob& j) {
  const H128Plan pl = h128_plan(j);
  if (pl.n_split <= 1) return kJoinRegionBytes;
  const size_t n = (size_t)(j.batch * j.n_q * (j.n_h / kH) * 2) * pl.n_split;  // (unit, split) slots
  return kJoinRegionBytes + n * (size_t)kH * 256 * sizeof(__nv_bfloat16) + n * kH * sizeof(float2) + 256;
}

cudaError_t launch_attend_h128(const AttendJob& j, void* ws, cudaStream_t s) {
  if (j.batch == 0 || j.n_q == 0 || j.n_h == 0) return cudaSuccess;
  H128Params p{};
  const H128Plan pl = h128_plan(j);
  p.idx = j.idx;
  p.q = static_cast<const __nv_bfloat16*>(j.q);
  p.kv = static_cast<const __nv_bfloat16*>(j.k);
  p.wkv = static_cast<const __nv_bfloat16*>(j.wk);
  p.o = j.o, p.lse = j.lse, p.out = j.out, p.out_bf16 = j.out_bf16;
  p.n_q = j.n_q, p.n_h = j.n_h, p.n_entries = j.n_entries, p.kv_stride = j.kv_stride, p.list_len = j.list_len;
  p.m = j.m, p.q_pos0 = j.q_pos0, p.q_pos = j.q_pos;
  p.n_split = pl.n_split;
  p.n_hg = (int)(j.n_h / kH);
  p.win = j.win;
  p.w_stride = j.w_stride, p.w_pos0 = j.w_pos0, p.wq_pos0 = j.wq_pos0, p.n_win = j.n_win;
  p.wq_pos = j.wq_pos, p.w_pos0s = j.w_pos0s;
  p.scale_log2 = j.scale * kLog2e;
  p.dev_status = j.dev_status;
  p.sink = j.sink;
  p.wait_cycles = grid_wait_cycles();
  const int64_t rows = j.batch * j.n_q;
  const int64_t units = rows * p.n_hg * 2;
  if (p.n_split > 1) {
    if (units > kMaxJoinUnits) return cudaErrorInvalidConfiguration;  // (the plan never splits those)
    const size_t n = (size_t)units * p.n_split;
    p.join_cnt = static_cast<uint32_t*>(ws);
    p.part_o = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + kJoinRegionBytes);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + kJoinRegionBytes +
                                          n * (size_t)kH * 256 * sizeof(__nv_bfloat16));
  }
  const uint64_t kv_rows = (uint64_t)(j.batch * j.kv_stride);
  p.k_rows = (int32_t)kv_rows;
  CUtensorMap tm_q, tm_k, tm_kg, tm_w, tm_wg;
  const uint32_t box_rows = kv_rows < (uint64_t)kT ? (uint32_t)kv_rows : (uint32_t)kT;
  if (!encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.q, kC, (uint64_t)(rows * j.n_h), kC * 2, 64, kH,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.k, kC, kv_rows, kC * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_kg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.k, kC, kv_rows, kC * 2, 64, 1,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  tm_w = tm_k, tm_wg = tm_kg;
  p.w_rows = p.k_rows;
  if (j.win) {
    const uint64_t w_rows = (uint64_t)(j.batch * j.w_stride);
    const uint32_t w_box = w_rows < (uint64_t)kT ? (uint32_t)w_rows : (uint32_t)kT;
    p.w_rows = (int32_t)w_rows;
    if (!encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.wk, kC, w_rows, kC * 2, 64, w_box,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&tm_wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.wk, kC, w_rows, kC * 2, 64, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int64_t grid = units * p.n_split;
  if (grid >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  auto run = [&](auto kernel) {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (r != cudaSuccess) return r;
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), (size_t)kSmemBytes, s, tm_q, tm_k, tm_kg, tm_w,
                      tm_wg, p);
  };
  cudaError_t e = j.mode == 0 ? run(attend_h128_kernel<0>) : run(attend_h128_kernel<1>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
