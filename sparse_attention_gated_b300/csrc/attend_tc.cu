// attend_tc.cu -- MQA core attention on the 5th-generation tensor cores for the
// three entry sources of the hybrid-attention forward:
//   mode 0, CSA: the entries listed by the top-k selector ("DeepSeek-V4 hybrid
//           attention" (trishampatil.com) section V.3: every query head attends
//           the same selected compressed entries, key = value = the entry);
//   mode 1, HCA: every visible entry, s < floor((t+1)/m') (same page, section VI);
//   mode 2, sliding window: raw rows max(0,t-n_win+1)..t, merged with the
//           compressed branch by log-sum-exp ("DeepSeek-V4: Anatomy..."
//           (modernaiengineering.com), "One query in a CSA layer", steps 4-5).
//
// Shapes: head dim c = 512, bf16 q / keys / values, query heads in groups of 64.
// One CTA owns one (query, group of 64 heads, split of the entry list).  All
// heads share one K (= V) row per entry, so per tile of 128 entries the work is
// two dense products, computed transposed so that the entries (then the head
// dimension) fill the 128 rows of the MMA and the 64 heads are its N:
//   S^T[e,h]  = sum_d K[e,d] Q[h,d]     M = 128 entries,  N = 64, K = 512
//   O^T[d,h] += sum_e V[e,d] P^T[e,h]   M = 128 dims x 4 chunks, N = 64, K = 128
// Both accumulate in TMEM (S^T: 2 x 64 columns, O^T: 4 x 64 columns), so the
// whole 64 x 512 float32 output of the CTA stays on chip until the epilogue.
// A tile is staged as 8 column slabs of [128 rows x 64 dims] in the 128-byte
// swizzle: the K-major A operand of S^T and, read with an MN-major
// descriptor, the A operand V^T of O^T.  The slabs stream through an 8-slot
// ring in the order K(0), K(1), V(0), K(2), V(1), ...: a tile's rows are
// loaded twice (the second time from L2 when V = K), which lets the next
// tile's loads and S^T overlap this tile's softmax within 227 KB of shared
// memory (the query group alone takes 64 KB).
//
// Warp roles (384 threads, one CTA per SM):
//   warps 0-2  producers: the query group by TMA once; entry slabs by TMA when
//              a tile is 128 consecutive rows, otherwise (index lists, ragged
//              last tile) gathered with 16-byte cp.async into the same
//              swizzled layout, rows without an entry zero-filled; for the
//              window merge, the compressed-branch output by one bulk copy.
//   warp 3     TMEM owner and MMA issuer (one elected thread).
//   warps 4-11 softmax and epilogue: two warps per TMEM lane quadrant, one
//              per half of the 64 heads; thread (e, half) owns TMEM lane e
//              (entry e of a tile, head-dim row e of an O^T chunk) for its
//              32 heads.
// Online softmax in base 2 with a lazy reference: the per-head reference
// m[h] only moves when some score exceeds it by more than 2^8, which a
// vote of the softmax warps detects; only then are the tile maxima reduced
// across the 128 entry lanes and the O^T accumulator rescaled.  Per-thread partial
// denominators are reduced across lanes once, at the end.
//
// Splits of one query's list write unnormalised partials (o, m, l) that a
// combine kernel merges.  Every wait is bounded (about 1 s): on expiry the
// kernel raises HYB_DEV_TIMEOUT in dev_status, lets its own copies and MMAs in
// flight land, frees TMEM and returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace hyb {

namespace {

constexpr int kProdWarps = 3, kMmaWarp = 3, kSoftWarp0 = 4, kSoftWarps = 8, kNumWarps = 12;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kHG = 64;                 // query heads per CTA (MMA N)
constexpr int kC = 512;                 // head dim c
constexpr int kTile = 128;              // entries per tile
constexpr int kSlabs = kC / 64;         // column slabs of 64 dims (128 bytes) per row
constexpr int kSlabBytes = kTile * 128;  // 16 KiB
constexpr int kQSlabBytes = kHG * 128;   // 8 KiB
constexpr int kMaxSplits = 64;         // splits of one (query, head group) list
// join counters at the start of the workspace: arrivals and departures of up to
// kMaxJoinUnits (query, head group) units; a launch with splits has at most one CTA
// per SM and at least two per unit
constexpr int kMaxJoinUnits = kNumSMs / 2;
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kSlabs * kQSlabBytes;
constexpr int kOffP = kOffKV + kSlabs * kSlabBytes;
constexpr int kOffRed = kOffP + kTile * kHG * 2;
// float scratch: red[2][64][4] (per-tile cross-quadrant exchange, double-buffered by
// tile parity: head-major so that one 16-byte load gets a head's four quadrants) and
// wt[8 warps][4][32] (each softmax warp's per-head table: reference, rescale factor,
// output coefficients)
constexpr int kRedFloats = 2 * 64 * 4 + 8 * 4 * 32;
constexpr int kOffBar = kOffRed + kRedFloats * 4;
constexpr int kNumBars = 1 + 2 * kSlabs + 2 + 2 + 1 + 1 + 2 + 1 + 1 + 1 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O^T: chunk ch at columns 64ch .. 64ch+63
constexpr uint32_t kTmemS = 256;  // S^T: buffer b at columns 256+64b ..
constexpr float kTau = 8.0f;      // lazy-reference threshold (log2 units): p <= 2^8
constexpr int kPrefetchAhead = 2;  // tiles whose rows are prefetched into L2 ahead of their loads
constexpr int kThreads = kNumWarps * 32;

static_assert(kSmemBytes <= 232448, "shared memory budget");

struct AtcParams {
  const int32_t* idx;       // mode 0: [rows][list_len]
  const __nv_bfloat16* k;   // gather sources, [batch][kv_stride][c]
  const __nv_bfloat16* v;
  float* o;                 // modes 0/1, one split: [rows][n_h][c]
  float* lse;               // [rows][n_h]
  __nv_bfloat16* part_o;    // modes 0/1, several splits: [rows][n_split][n_hg][4][64][128] (chunk-major)
  uint32_t* join_cnt;       // modes 0/1, several splits: [2][units] arrivals and departures (start and end at 0)
  float2* part_ml;          // [rows][n_split][n_h] (reference m in log2 units, denominator)
  const float* o_in;        // mode 2
  const float* lse_in;
  void* out;
  float* lse_out;
  int out_bf16;
  int64_t n_q, n_h, n_entries, kv_stride, list_len, m, q_pos0, kv_pos0, n_win;
  int n_split, n_hg, alias;
  // modes 0/1 with a fused window merge: the last split of each (query, head group) attends
  // the query's window of raw rows kw [batch][w_stride][c] (row 0 = absolute position w_pos0;
  // the rows are keys and values), and the join writes the merged `out` and the union's lse
  int win;
  const __nv_bfloat16* kw;
  int64_t w_stride, w_pos0, wq_pos0;
  // optional positions in device memory (read after the grid-dependency wait): per-query
  // positions of the call (modes 1/2) and of the fused window, per-sequence kv_pos0 of the
  // window rows (mode 2) and of the fused window's
  const int64_t* q_pos;
  const int64_t* kv_pos0s;
  const int64_t* wq_pos;
  const int64_t* w_pos0s;
  float scale_log2;
  int32_t* dev_status;
  long long wait_cycles;  // bound of the split join's wait (SM clock cycles)
};

struct AtcWork {
  int64_t bq, b, j, hg, sp;
  int64_t L;     // list length of this query
  int64_t row0;  // modes 1/2: global row of list position 0
  const int32_t* list;
  int64_t tb, te;  // this split's tiles
  bool win;        // this split is the fused window (contiguous rows of kw)
};

template <int MODE>
__device__ __forceinline__ AtcWork atc_work(const AtcParams& p) {
  AtcWork w;
  const int64_t id = blockIdx.x;  // split fastest: the splits of a unit are consecutive CTAs
  w.sp = id % p.n_split;
  w.hg = (id / p.n_split) % p.n_hg;
  w.bq = id / ((int64_t)p.n_hg * p.n_split);
  w.b = w.bq / p.n_q;
  w.j = w.bq % p.n_q;
  const bool report = w.hg == 0 && threadIdx.x == 0;
  w.list = nullptr;
  w.row0 = 0;
  w.win = false;
  if (MODE != 2 && p.win && w.sp == p.n_split - 1) {
    // the fused window: raw rows max(0, tw-n_win+1) .. tw of kw
    const int64_t tw = query_pos(p.wq_pos, p.wq_pos0, w.bq, w.j);
    const int64_t kvp = p.w_pos0s ? __ldg(p.w_pos0s + w.b) : p.w_pos0;
    int64_t first;
    w.win = true;
    w.L = window_rows(tw, p.n_win, kvp, p.w_stride, &first, p.dev_status, report);
    w.row0 = w.b * p.w_stride + first;
    w.tb = 0;
    w.te = (w.L + kTile - 1) / kTile;
    return w;
  }
  const int64_t t = MODE == 0 ? 0 : query_pos(p.q_pos, p.q_pos0, w.bq, w.j);
  if constexpr (MODE == 0) {
    w.L = p.list_len;
    w.list = p.idx + w.bq * p.list_len;
  } else if constexpr (MODE == 1) {
    w.L = visible_checked(t, p.m, p.n_entries, p.dev_status, report && w.sp == 0);
    w.row0 = w.b * p.kv_stride;
  } else {
    const int64_t kvp = p.kv_pos0s ? __ldg(p.kv_pos0s + w.b) : p.kv_pos0;
    int64_t first;
    w.L = window_rows(t, p.n_win, kvp, p.kv_stride, &first, p.dev_status, report && w.sp == 0);
    w.row0 = w.b * p.kv_stride + first;
    // (split window merges divide the output dims, not the rows: every split sees the window)
    w.tb = 0;
    w.te = (w.L + kTile - 1) / kTile;
    return w;
  }
  const int64_t T = (w.L + kTile - 1) / kTile;
  const int64_t S = p.n_split - (MODE != 2 && p.win ? 1 : 0);  // splits of the compressed list
  w.tb = w.sp * T / S;
  w.te = (w.sp + 1) * T / S;
  return w;
}

// Global row of list position pos, or -1 when the position holds no entry.
template <int MODE>
__device__ __forceinline__ int64_t atc_row(const AtcParams& p, const AtcWork& w, int64_t pos, bool report) {
  if (pos >= w.L) return -1;
  if (MODE != 2 && w.win) return w.row0 + pos;
  if constexpr (MODE == 0) {
    const int32_t s = __ldg(w.list + pos);
    if (s == -1) return -1;
    if (s < -1 || s >= p.n_entries) {
      if (report) flag_status(p.dev_status, HYB_DEV_BAD_INDEX);
      return -1;
    }
    return w.b * p.kv_stride + s;
  } else {
    return w.row0 + pos;
  }
}

// Load group G of 2n (n tiles) in streaming order K(0), K(1), V(0), K(2), V(1),
// ..., K(n-1), V(n-2), V(n-1): returns the tile and whether it is the V pass.
__device__ __forceinline__ int64_t atc_group(int64_t G, int64_t ngroups, bool& is_v) {
  if (G == 0) {
    is_v = false;
    return 0;
  }
  if (G == ngroups - 1) {
    is_v = true;
    return ngroups / 2 - 1;
  }
  is_v = (G & 1) == 0;
  return is_v ? G / 2 - 1 : (G + 1) / 2;
}

// Warp that gathers slab g.  Index lists (mode 0) rotate over the producer
// warps: each warp waits on some slot every third slab and slots are released
// in slab order, so no warp waits on a slot more than one phase ahead.  The
// contiguous modes gather only a ragged last tile, after TMA tiles that warp 0
// issued alone; warp 0 also gathers so that every slot's phases are waited in
// order by one warp.  A list shorter than a tile has no TMA tile at all.
template <int MODE>
__device__ __forceinline__ int atc_gather_warp(int64_t g, int64_t list_len, bool contiguous) {
  return (!contiguous || list_len < kTile) ? (int)(g % kProdWarps) : 0;
}

// Reduce 32 per-lane values (one per head) across the 32 lanes of a warp by
// recursive halving: after the five exchange steps lane l holds the reduction
// for value l.  31 shuffles instead of 160.
template <bool MAX>
__device__ __forceinline__ float transpose_reduce32(float (&a)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float lo = a[i], hi = a[i + o];
      const float send = up ? lo : hi;
      const float keep = up ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      a[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return a[0];
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                     AtcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + kOffQ;
  uint8_t* kv_s = smem + kOffKV;
  uint8_t* p_s = smem + kOffP;
  float* red = reinterpret_cast<float*>(smem + kOffRed);  // [2][64][4]
  float* wtab = red + 2 * 64 * 4;                           // [8][4][32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + kSlabs;
  uint64_t* s_full = kv_empty + kSlabs;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* sm_sync = o_done + 1;  // [2]: one per head half (4 softmax warps each)
  uint64_t* fin = sm_sync + 2;
  uint64_t* oin_full = fin + 1;
  uint64_t* q_free = oin_full + 1;  // the last products that read the query are done
  uint64_t* sm_all = q_free + 1;     // all softmax warps (the split join)
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // positions in device memory may have been written by the previous kernel: read them after the wait
  if (p.q_pos != nullptr || p.kv_pos0s != nullptr || p.wq_pos != nullptr || p.w_pos0s != nullptr) pdl_wait();
  const AtcWork W = atc_work<MODE>(p);
  const int64_t ntiles = W.te - W.tb;
  // K = V and one tile: O^T reads the K slabs still in the ring (no V group);
  // otherwise the V slabs are loaded again after the next tile's K (see above)
  const bool contig = MODE != 0 || W.win;  // rows are consecutive (TMA tiles where whole)
  const bool reuse = (p.alias || W.win) && ntiles == 1;
  const int64_t ngroups = reuse ? 1 : 2 * ntiles;
  // O^T chunks (128 dims each) this CTA computes: a split window merge takes 4/n_split of them
  const int ch0 = MODE == 2 ? (int)W.sp * (4 / p.n_split) : 0;
  const int ch1 = MODE == 2 ? ch0 + 4 / p.n_split : 4;

  // the first group's loads are issued by the thread that initialises the
  // barriers, before the CTA-wide setup sync (overlapping the TMEM allocation)
  const bool pre_k = contig && ntiles > 0 && (W.tb + 1) * kTile <= W.L;
  const CUtensorMap* tm_k0 = W.win ? &tm_w : &tm_k;  // the key rows' map
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < kSlabs; ++s) tc::mbar_init(&kv_full[s], 1), tc::mbar_init(&kv_empty[s], 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&s_full[i], 1), tc::mbar_init(&s_empty[i], kSoftWarps);
    tc::mbar_init(p_full, kSoftWarps);
    tc::mbar_init(o_done, 1);
    tc::mbar_init(&sm_sync[0], kSoftThreads / 2);
    tc::mbar_init(&sm_sync[1], kSoftThreads / 2);
    tc::mbar_init(fin, 1);
    tc::mbar_init(oin_full, 1);
    tc::mbar_init(q_free, 1);
    tc::mbar_init(sm_all, kSoftThreads);
    *s_abort = 0;
    tc::fence_barrier_init();
    pdl_wait();  // the loads below may read what the previous kernel wrote
    if (ntiles > 0) {
      tc::prefetch_tmap(&tm_q);
      tc::mbar_arrive_expect_tx(q_full, kSlabs * kQSlabBytes);
      const int32_t qrow = (int32_t)(W.bq * p.n_h + W.hg * kHG);
      for (int s = 0; s < kSlabs; ++s) tc::tma_load_2d(q_s + s * kQSlabBytes, &tm_q, q_full, 64 * s, qrow);
    }
    if (pre_k) {
      tc::prefetch_tmap(tm_k0);
      for (int s = 0; s < kSlabs; ++s) {
        tc::mbar_arrive_expect_tx(&kv_full[s], kSlabBytes);
        tc::tma_load_2d(kv_s + s * kSlabBytes, tm_k0, &kv_full[s], 64 * s, (int32_t)(W.row0 + W.tb * kTile));
      }
    }
    if (MODE != 0 && !W.win) tc::prefetch_tmap(&tm_v);
  }
  if (warp == kMmaWarp) tc::tmem_alloc(s_tmem, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // (before it: shared memory, TMEM and parameters only, except thread 0's loads above)
  pdl_trigger();

  bool sm_ok = false;  // softmax warps: the main loop and epilogue completed
  if (warp < kProdWarps) {
    // ================================================================ producers
    bool ok = true;
    int64_t tma_u[kSlabs];  // last use count of each slot filled by TMA (for the drain on abort)
#pragma unroll
    for (int s = 0; s < kSlabs; ++s) tma_u[s] = pre_k ? 0 : -1;
    // L2 prefetch of the entry rows kPrefetchAhead tiles ahead of the K group being
    // loaded, so the loads that later fill the ring pay L2 rather than HBM latency
    auto prefetch_tile = [&](int64_t i) {
      if (i >= W.te) return;
      if (contig) {
        if (warp == 0 && lane == 0) {
          const int64_t n = std::min<int64_t>(kTile, W.L - i * kTile);
          tc::prefetch_l2((W.win ? p.kw : p.k) + (W.row0 + i * kTile) * kC, (uint32_t)(n * kC * 2));
        }
      } else if (warp == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int64_t row = atc_row<MODE>(p, W, i * kTile + lane + 32 * r, false);
          if (row >= 0) tc::prefetch_l2(p.k + row * kC, kC * 2);
        }
      }
    };
    for (int64_t a = 1; a <= kPrefetchAhead; ++a) prefetch_tile(W.tb + a);
    int64_t g = pre_k ? kSlabs : 0;  // slab sequence number
    for (int64_t G = pre_k ? 1 : 0; G < ngroups && ok; ++G) {
      bool is_v;
      const int64_t li = atc_group(G, ngroups, is_v);
      const int64_t i = W.tb + li;
      if (!is_v && li > 0) prefetch_tile(i + kPrefetchAhead);
      const bool tma_tile = contig && (i + 1) * kTile <= W.L;
      int64_t rows[4];
      if (!tma_tile) {
#pragma unroll
        for (int r = 0; r < 4; ++r) rows[r] = atc_row<MODE>(p, W, i * kTile + lane + 32 * r, warp == 0 && !is_v);
      }
      const CUtensorMap* tm = W.win ? &tm_w : (is_v ? &tm_v : &tm_k);
      const __nv_bfloat16* src = W.win ? p.kw : (is_v ? p.v : p.k);
      const uint32_t par = (uint32_t)(G & 1) ^ 1u;  // wait for the release of the slot's previous use
      for (int s = 0; s < kSlabs; ++s, ++g) {
        uint8_t* dst = kv_s + s * kSlabBytes;
        if (tma_tile) {
          if (warp == 0) {
            int okl = 1;
            if (lane == 0) {
              okl = tc::mbar_wait(&kv_empty[s], par, s_abort, 1);
              if (okl) {
                tc::mbar_arrive_expect_tx(&kv_full[s], kSlabBytes);
                tc::tma_load_2d(dst, tm, &kv_full[s], 64 * s, (int32_t)(W.row0 + i * kTile));
                tma_u[s] = G;
              }
            }
            ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
            if (!ok) break;
          }
        } else if (atc_gather_warp<MODE>(g, W.L, contig) == warp) {
          int okl = 1;
          if (lane == 0) okl = tc::mbar_wait(&kv_empty[s], par, s_abort, 2);
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          if (!ok) break;
          // eight lanes per row, one 16-byte chunk each: every instruction moves four whole
          // 128-byte row pieces (entry e = 4*i + lane/8 takes its row from lane e % 32, value e / 32)
          const uint32_t dbase = tc::smem_u32(dst);
          const int c16 = lane & 7;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = 4 * i + (lane >> 3);
            const int32_t row = __shfl_sync(0xffffffffu, (int32_t)rows[i >> 3], (4 * i + (lane >> 3)) & 31);
            const bool have = row >= 0;
            const __nv_bfloat16* rsrc = src + (int64_t)(have ? row : 0) * kC + s * 64 + c16 * 8;
            const uint32_t dchunk = dbase + (uint32_t)((e >> 3) * 1024 + (e & 7) * 128 + ((c16 ^ (e & 7)) << 4));
            tc::cp_async16(dchunk, rsrc, have ? 16u : 0u);
          }
          // the slab is complete once every lane's copies have landed; nobody waits here
          tc::cp_async_arrive_on(&kv_full[s]);
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&kv_full[s]);
        }
      }
    }
    tc::cp_async_wait_all();  // this thread's copies have landed before it leaves
    bool oin_issued = false;
    if constexpr (MODE == 2) {
      if (p.n_split > 1) {
        // this split's dims of the compressed-branch output, [64 heads][D], into the query
        // region once the last products that read the query are done
        if (ok && warp == 0 && p.o_in != nullptr) {
          int okl = 1;
          if (lane == 0) {
            if (ntiles > 0) okl = tc::mbar_wait(q_free, 0, s_abort, 15);
            if (okl) {
              const int D = kC / p.n_split;
              tc::mbar_arrive_expect_tx(oin_full, (uint32_t)(kHG * D * 4));
              const float* src = p.o_in + (W.bq * p.n_h + W.hg * kHG) * kC + W.sp * D;
              for (int h = 0; h < kHG; ++h)
                tc::bulk_load(q_s + h * D * 4, src + (int64_t)h * kC, (uint32_t)(D * 4), oin_full);
              oin_issued = true;
            }
          }
          ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
          oin_issued = __shfl_sync(0xffffffffu, (int)oin_issued, 0) != 0;
        }
      } else if (ok && warp == 0 && p.o_in != nullptr && ntiles > 0) {
        // the compressed-branch output of this query's heads, into the ring once the last products are done
        int okl = 1;
        if (lane == 0) {
          const uint32_t lastpar = (uint32_t)((ngroups - 1) & 1);
          for (int s = 0; s < kSlabs && okl; ++s) okl = tc::mbar_wait(&kv_empty[s], lastpar, s_abort, 13);
          if (okl) {
            tc::mbar_arrive_expect_tx(oin_full, kSlabs * kSlabBytes);
            const float* src = p.o_in + (W.bq * p.n_h + W.hg * kHG) * kC;
            for (int s = 0; s < kSlabs; ++s)
              tc::bulk_load(kv_s + s * kSlabBytes, src + s * (kSlabBytes / 4), kSlabBytes, oin_full);
            oin_issued = true;
          }
        }
        ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
        oin_issued = __shfl_sync(0xffffffffu, (int)oin_issued, 0) != 0;
      }
    }
    if (!ok && warp == 0 && lane == 0) {
      // let this thread's TMA copies in flight land before the CTA can exit
      for (int s = 0; s < kSlabs; ++s)
        if (tma_u[s] >= 0) tc::mbar_wait_drain(&kv_full[s], (uint32_t)(tma_u[s] & 1));
      if (ntiles > 0) tc::mbar_wait_drain(q_full, 0);
    }
    if (oin_issued && *s_abort && lane == 0) tc::mbar_wait_drain(oin_full, 0);
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    // Groups in load order: K(0), K(1), V(0), K(2), V(1), ..., V(n-1).  S^T of the
    // next tile is issued before O^T of this one, so the next tile's loads and
    // products overlap this tile's softmax.
    if (tc::elect_one()) {
      bool ok = ntiles == 0 || tc::mbar_wait(q_full, 0, s_abort, 3);
      constexpr uint32_t idS = tc::make_idesc(1, 1, 0, 0, 128, kHG);  // A = K (K-major), B = Q (K-major)
      constexpr uint32_t idO = tc::make_idesc(1, 1, 1, 1, 128, kHG);  // A = V^T (MN-major), B = P^T (MN-major)
      const uint32_t q_addr = tc::smem_u32(q_s), kv_addr = tc::smem_u32(kv_s), p_addr = tc::smem_u32(p_s);
      for (int64_t G = 0; G < ngroups && ok; ++G) {
        bool is_v;
        const int64_t li = atc_group(G, ngroups, is_v);
        const uint32_t par = (uint32_t)(G & 1);
        if (!is_v) {
          const int sb = (int)(li & 1);
          if (!(ok = tc::mbar_wait(&s_empty[sb], (uint32_t)((li >> 1) & 1) ^ 1u, s_abort, 4))) break;
          const uint32_t dS = tmem + kTmemS + (uint32_t)(sb * kHG);
          for (int s = 0; s < kSlabs; ++s) {
            if (!(ok = tc::mbar_wait(&kv_full[s], par, s_abort, 5))) break;
            tc::fence_proxy_async_smem();  // gathered slabs were written through the generic proxy
            tc::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_f16(dS, tc::desc_kmajor_sw128(kv_addr + s * kSlabBytes + 32 * kk),
                          tc::desc_kmajor_sw128(q_addr + s * kQSlabBytes + 32 * kk), idS, (s | kk) ? 1u : 0u);
            if (!reuse) tc::mma_commit(&kv_empty[s]);  // the slot is free once these products are done
          }
          if (!ok) break;
          tc::mma_commit(&s_full[sb]);
          if (li == ntiles - 1) tc::mma_commit(q_free);
          if (reuse) {
            // O^T from the same slabs (they are V too), then release them
            if (!(ok = tc::mbar_wait(p_full, 0, s_abort, 6))) break;
            tc::tc_fence_after();
            for (int ch = 0; ch < 4; ++ch) {
              const uint32_t a0 = kv_addr + (uint32_t)(2 * ch * kSlabBytes);
              if (ch >= ch0 && ch < ch1) {
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                  tc::mma_f16(tmem + kTmemO + (uint32_t)(ch * kHG),
                              tc::desc_mnmajor_sw128(a0 + ks * 2048, kSlabBytes, 1024),
                              tc::desc_mnmajor_sw128(p_addr + ks * 2048, 16, 1024), idO, ks > 0 ? 1u : 0u);
              }
              tc::mma_commit(&kv_empty[2 * ch]);
              tc::mma_commit(&kv_empty[2 * ch + 1]);
            }
            tc::mma_commit(o_done);
          }
        } else {
          if (!(ok = tc::mbar_wait(p_full, (uint32_t)(li & 1), s_abort, 6))) break;
          tc::tc_fence_after();
          for (int ch = 0; ch < 4; ++ch) {
            if (!(ok = tc::mbar_wait(&kv_full[2 * ch], par, s_abort, 7))) break;
            if (!(ok = tc::mbar_wait(&kv_full[2 * ch + 1], par, s_abort, 7))) break;
            tc::fence_proxy_async_smem();
            tc::tc_fence_after();
            // V^T chunk ch: dims 128ch.. (slabs 2ch, 2ch+1: leading offset one slab), entries along K
            // in 8-row groups 1024 bytes apart; P^T has one 64-head group (leading offset unused)
            const uint32_t a0 = kv_addr + (uint32_t)(2 * ch * kSlabBytes);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
              tc::mma_f16(tmem + kTmemO + (uint32_t)(ch * kHG),
                          tc::desc_mnmajor_sw128(a0 + ks * 2048, kSlabBytes, 1024),
                          tc::desc_mnmajor_sw128(p_addr + ks * 2048, 16, 1024), idO, (li > 0 || ks > 0) ? 1u : 0u);
            tc::mma_commit(&kv_empty[2 * ch]);
            tc::mma_commit(&kv_empty[2 * ch + 1]);
          }
          if (!ok) break;
          tc::mma_commit(o_done);
        }
      }
      // every MMA issued above has completed once `fin` flips
      tc::mma_commit(fin);
      tc::mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax + epilogue
    // Warp w owns TMEM lane quadrant w % 4 (entries / head-dim rows 32(w%4) ..)
    // and head half hh = (w - 4) / 4 (heads 32hh .. 32hh+31).  The four warps
    // of a half exchange per-head values through shared memory and meet on
    // their own barrier; the halves never wait on each other.
    const int q4 = warp & 3;
    const int hh = (warp - kSoftWarp0) >> 2;
    const int e = q4 * 32 + lane;  // tile entry / O^T chunk row owned by this thread
    const int h0 = hh * 32;        // first head of this thread
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    uint64_t* my_sync = &sm_sync[hh];
    uint32_t sync_phase = 0;
    auto hsync = [&]() -> bool {
      tc::mbar_arrive(my_sync);
      const bool r = tc::mbar_wait(my_sync, sync_phase, s_abort, 9);
      sync_phase ^= 1u;
      return r;
    };
    float lp[32];  // partial denominators of this entry lane, per head
#pragma unroll
    for (int h = 0; h < 32; ++h) lp[h] = 0.f;
    // This warp's table, one column per head of its half; lane l owns head h0+l:
    //   wt_m: softmax reference (log2 units), wt_a: rescale factor of the tile,
    //   wt_cw / wt_cc: output coefficients of the accumulator / of o_in.
    // Every warp of a half computes the same values from the same inputs.
    float* wt_m = wtab + (warp - kSoftWarp0) * 128;
    float* wt_a = wt_m + 32;
    float* wt_cw = wt_m + 64;
    float* wt_cc = wt_m + 96;
    wt_m[lane] = -INFINITY;
    __syncwarp();
    bool ok = true;

    for (int64_t li = 0; li < ntiles && ok; ++li) {
      const int64_t i = W.tb + li;
      const int sb = (int)(li & 1);
      if (!(ok = tc::mbar_wait(&s_full[sb], (uint32_t)((li >> 1) & 1), s_abort, 8))) break;
      tc::tc_fence_after();
      const uint32_t sS = tmem + lane_base + kTmemS + (uint32_t)(sb * kHG + h0);
      const bool valid = atc_row<MODE>(p, W, i * kTile + e, false) >= 0;
      float sv[32];
      auto load_scores = [&]() {
        tc::tmem_ld32(sS, sv);
        tc::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) sv[h] = valid ? sv[h] * p.scale_log2 : -INFINITY;
      };
      load_scores();
      // tile maximum of each head: over this warp's 32 entries (lane l gets head h0+l),
      // then over the 4 quadrants through shared memory
      float* redb = red + sb * 256;
      redb[(h0 + lane) * 4 + q4] = transpose_reduce32<true>(sv, lane);
      if (!(ok = hsync())) break;
      // lazy reference of head h0+lane: moves only when the tile maximum exceeds it by
      // more than 2^kTau (or there was none)
      {
        const float4 r4 = *reinterpret_cast<const float4*>(redb + (h0 + lane) * 4);
        const float tmax = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
        const float mo = wt_m[lane];
        const bool mv = tmax > mo + kTau || (mo == -INFINITY && tmax != -INFINITY);
        wt_a[lane] = mv ? exp2f(mo - tmax) : 1.f;  // 0 when there was no reference
        wt_m[lane] = mv ? tmax : mo;
      }
      const bool moved = __any_sync(0xffffffffu, wt_a[lane] != 1.f);
      __syncwarp();
      bool odone = false;
      if (moved) {
        float al[32];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 a4 = *reinterpret_cast<const float4*>(wt_a + 4 * x);
          al[4 * x] = a4.x, al[4 * x + 1] = a4.y, al[4 * x + 2] = a4.z, al[4 * x + 3] = a4.w;
        }
#pragma unroll
        for (int h = 0; h < 32; ++h) lp[h] *= al[h];
        if (li > 0) {
          // rescale this thread's O^T lane (its heads, every chunk) once the previous products are done
          if (!(ok = tc::mbar_wait(o_done, (uint32_t)((li - 1) & 1), s_abort, 10))) break;
          odone = true;
          tc::tc_fence_after();
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            float v[32];
            const uint32_t ta = tmem + lane_base + kTmemO + (uint32_t)(ch * kHG + h0);
            tc::tmem_ld32(ta, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int y = 0; y < 32; ++y) v[y] *= al[y];
            tc::tmem_st32(ta, v);
          }
          tc::tmem_st_wait();
        }
      }
      // probabilities of this entry for this thread's heads: 64 bytes of row e of P^T (bf16)
      load_scores();  // the reduction consumed the registers
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&s_empty[sb]);
      uint32_t pk[16];
      if (valid) {
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 m4 = *reinterpret_cast<const float4*>(wt_m + 4 * x);
          const float p0 = exp2f(sv[4 * x] - m4.x), p1 = exp2f(sv[4 * x + 1] - m4.y);
          const float p2 = exp2f(sv[4 * x + 2] - m4.z), p3 = exp2f(sv[4 * x + 3] - m4.w);
          lp[4 * x] += p0, lp[4 * x + 1] += p1, lp[4 * x + 2] += p2, lp[4 * x + 3] += p3;
          pk[2 * x] = pack_bf16x2(p0, p1);
          pk[2 * x + 1] = pack_bf16x2(p2, p3);
        }
      } else {
#pragma unroll
        for (int x = 0; x < 16; ++x) pk[x] = 0u;
      }
      if (li > 0 && !odone) {
        if (!(ok = tc::mbar_wait(o_done, (uint32_t)((li - 1) & 1), s_abort, 11))) break;
      }
      uint8_t* prow = p_s + (e >> 3) * 1024 + (e & 7) * 128;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int c16 = hh * 4 + x;
        *reinterpret_cast<uint4*>(prow + ((c16 ^ (e & 7)) << 4)) =
            make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(p_full);
    }

    // ---------------------------------------------------------------- epilogue
    // denominators: reduce the per-entry partial sums of every head across the 128 entry lanes
    float* redl = red + (int)(ntiles & 1) * 256;  // the buffer the last tile did not use
    if (ok) {
      redl[(h0 + lane) * 4 + q4] = transpose_reduce32<false>(lp, lane);
      ok = hsync();
    }
    // output coefficients of head h0+lane (acc multiplier cw, o_in multiplier cc), its lse
    if (ok) {
      const float4 r4 = *reinterpret_cast<const float4*>(redl + (h0 + lane) * 4);
      const float l = (r4.x + r4.y) + (r4.z + r4.w);
      const float mm = wt_m[lane];
      const int64_t H = W.hg * kHG + h0 + lane;
      const float lse2 = l > 0.f ? mm + __log2f(l) : -INFINITY;  // log2 of the denominator
      float cw, cc = 0.f;
      if constexpr (MODE == 2) {
        // one softmax over the union of the window and the compressed set
        const float lse_w = lse2 * kLn2;
        const float lse_c = p.lse_in ? p.lse_in[W.bq * p.n_h + H] : -INFINITY;
        const float M = fmaxf(lse_w, lse_c);
        float Lse = -INFINITY;
        cw = 0.f;
        if (M != -INFINITY) {
          const float ec = lse_c == -INFINITY ? 0.f : expf(lse_c - M);
          const float ew = lse_w == -INFINITY ? 0.f : expf(lse_w - M);
          const float den = ec + ew;
          cc = ec / den;
          cw = ew / (den * (l > 0.f ? l : 1.f));  // the accumulator is unnormalised
          Lse = M + logf(den);
        }
        if (q4 == 0 && W.sp == 0 && p.lse_out) p.lse_out[W.bq * p.n_h + H] = Lse;
      } else if (p.n_split > 1) {
        cw = 1.f;
        const float2 ml = make_float2(l > 0.f ? mm : -INFINITY, l);
        if (q4 == 0) {
          p.part_ml[(W.bq * p.n_split + W.sp) * p.n_h + H] = ml;
        }
      } else {
        cw = l > 0.f ? 1.f / l : 0.f;
        if (q4 == 0) p.lse[W.bq * p.n_h + H] = lse2 * kLn2;
      }
      wt_cw[lane] = cw;
      wt_cc[lane] = cc;
      __syncwarp();
    }
    if (ok && ntiles > 0) {
      ok = tc::mbar_wait(o_done, (uint32_t)((ntiles - 1) & 1), s_abort, 12);
      tc::tc_fence_after();
    }
    sm_ok = ok;
    if constexpr (MODE == 2) {
      if (ok && p.o_in != nullptr) ok = tc::mbar_wait(oin_full, 0, s_abort, 14);
    }
    if (MODE == 2 && ok && p.n_split > 1) {
      // split window merge: this CTA's chunks, merged with the staged o_in slice
      // [64 heads][D] (query region), stored straight from registers (lanes along dims)
      const int D = kC / p.n_split;
      const float* oin = reinterpret_cast<const float*>(q_s);
      const bool have_oin = p.o_in != nullptr;
      const int64_t orow = (W.bq * p.n_h + W.hg * kHG + h0) * kC;
#pragma unroll 1
      for (int ch = ch0; ch < ch1; ++ch) {
        float v[32], cw[32], oc[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(ch * kHG + h0), v);
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] = 0.f;
        }
        const int dl = (ch - ch0) * 128 + e;  // dim within the slice
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 a = *reinterpret_cast<const float4*>(wt_cw + 4 * x);
          cw[4 * x] = a.x, cw[4 * x + 1] = a.y, cw[4 * x + 2] = a.z, cw[4 * x + 3] = a.w;
          const float4 b = *reinterpret_cast<const float4*>(wt_cc + 4 * x);
          oc[4 * x] = b.x, oc[4 * x + 1] = b.y, oc[4 * x + 2] = b.z, oc[4 * x + 3] = b.w;
        }
#pragma unroll
        for (int y = 0; y < 32; ++y) oc[y] = (have_oin && oc[y] != 0.f) ? oc[y] * oin[(h0 + y) * D + dl] : 0.f;
        if (ntiles > 0) tc::tmem_ld_wait();
        const int64_t o0 = orow + ch * 128 + e;
        if (p.out_bf16) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + o0;
#pragma unroll
          for (int y = 0; y < 32; ++y) out[(int64_t)y * kC] = __float2bfloat16_rn(fmaf(cw[y], v[y], oc[y]));
        } else {
          float* out = static_cast<float*>(p.out) + o0;
#pragma unroll
          for (int y = 0; y < 32; ++y) out[(int64_t)y * kC] = fmaf(cw[y], v[y], oc[y]);
        }
      }
    } else if (MODE != 2 && ok && p.n_split > 1) {
      // split partial (unnormalised O, rounded to bf16 like the probabilities that made it):
      // chunk by chunk, this half's [32 heads][128] piece is staged in the free ring and
      // bulk-stored at once into the unit's chunk-major partial [4 chunks][64 heads][128]
      __nv_bfloat16* piece0 = reinterpret_cast<__nv_bfloat16*>(kv_s) + hh * (4 * 32 * 128);
      __nv_bfloat16* dst0 = p.part_o + ((W.bq * p.n_split + W.sp) * p.n_hg + W.hg) * (int64_t)(kHG * kC);
#pragma unroll 1
      for (int ch = 0; ch < 4 && ok; ++ch) {
        float v[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(ch * kHG + h0), v);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] = 0.f;
        }
        __nv_bfloat16* piece = piece0 + ch * (32 * 128);
#pragma unroll
        for (int y = 0; y < 32; ++y) piece[y * 128 + e] = __float2bfloat16_rn(v[y]);
        tc::fence_proxy_async_smem();
        ok = hsync();
        if (ok && q4 == 0 && lane == 0) {
          tc::bulk_store(dst0 + (int64_t)(ch * kHG + h0) * 128, piece, 32 * 128 * 2);
          tc::bulk_commit();
        }
      }
      if (q4 == 0 && lane == 0) {
        tc::bulk_wait_all();  // the partial is in global memory before this split counts itself done
        tc::fence_proxy_async_global();
      }
    } else if (ok) {
      // O^T (TMEM) -> this half's 32 rows of [64 heads][512] in shared memory -> one bulk store.
      // Staging: float32 in the free K/V ring (in place over the staged o_in for a float32
      // window merge), bf16 window-merge output in the free query region.
      const bool out_bf16 = MODE == 2 && p.out_bf16;
      float* stage32 = reinterpret_cast<float*>(kv_s) + h0 * kC;
      __nv_bfloat16* stage16 = reinterpret_cast<__nv_bfloat16*>(q_s) + h0 * kC;
      const float* oin = reinterpret_cast<const float*>(kv_s) + h0 * kC;  // staged o_in (window merge)
      const bool have_oin = MODE == 2 && p.o_in != nullptr;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        // every load of the chunk first (stores to shared memory in between would serialise them)
        float v[32], cw[32], oc[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(ch * kHG + h0), v);
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] = 0.f;
        }
        const int d = ch * 128 + e;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const float4 a = *reinterpret_cast<const float4*>(wt_cw + 4 * x);
          cw[4 * x] = a.x, cw[4 * x + 1] = a.y, cw[4 * x + 2] = a.z, cw[4 * x + 3] = a.w;
        }
        if (have_oin) {
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float4 b = *reinterpret_cast<const float4*>(wt_cc + 4 * x);
            oc[4 * x] = b.x, oc[4 * x + 1] = b.y, oc[4 * x + 2] = b.z, oc[4 * x + 3] = b.w;
          }
#pragma unroll
          for (int y = 0; y < 32; ++y) oc[y] = oc[y] != 0.f ? oc[y] * oin[y * kC + d] : 0.f;
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) oc[y] = 0.f;
        }
        if (ntiles > 0) tc::tmem_ld_wait();
#pragma unroll
        for (int y = 0; y < 32; ++y) {
          const float r = fmaf(cw[y], v[y], oc[y]);
          if (out_bf16)
            stage16[y * kC + d] = __float2bfloat16_rn(r);
          else
            stage32[y * kC + d] = r;
        }
      }
      tc::fence_proxy_async_smem();
      ok = hsync();
      if (ok && q4 == 0 && lane == 0) {
        void* dst;
        if constexpr (MODE == 2)
          dst = out_bf16 ? static_cast<void*>(static_cast<__nv_bfloat16*>(p.out) + (W.bq * p.n_h + W.hg * kHG + h0) * kC)
                         : static_cast<void*>(static_cast<float*>(p.out) + (W.bq * p.n_h + W.hg * kHG + h0) * kC);
        else
          dst = p.o + (W.bq * p.n_h + W.hg * kHG + h0) * kC;
        const uint32_t bytes = 32 * kC * (out_bf16 ? 2 : 4);
        const uint8_t* src = out_bf16 ? reinterpret_cast<const uint8_t*>(stage16) : reinterpret_cast<const uint8_t*>(stage32);
        for (uint32_t off = 0; off < bytes; off += 16384)
          tc::bulk_store(static_cast<uint8_t*>(dst) + off, src + off, 16384);
        tc::bulk_commit();
        tc::bulk_wait_read();
      }
    }
    if (MODE != 2 && p.n_split > 1) {
      // Join the splits of this (query, head group) through L2: once every split has
      // counted itself done, split sp merges items [sp*N/S, (sp+1)*N/S) of the unit's
      // N = 64 heads x 128 float4 quads from the S partials (all CTAs of a launch with
      // splits are resident at once: at most one per SM).  Every wait is bounded.
      const int S = p.n_split;
      const int ts = (int)threadIdx.x - kSoftWarp0 * 32;
      uint32_t jphase = 0;
      auto all_sync = [&]() -> bool {
        tc::mbar_arrive(sm_all);
        const bool r = tc::mbar_wait(sm_all, jphase, s_abort, 17);
        jphase ^= 1u;
        return r;
      };
      ok = ok && all_sync();
      if (ok && ts == 0) {
        const int64_t unit = W.bq * p.n_hg + W.hg;
        uint32_t* cnt = p.join_cnt + unit;
        uint32_t* dep = p.join_cnt + kMaxJoinUnits + unit;
        __threadfence();
        atomicAdd(cnt, 1u);
        const long long t0 = clock64();
        bool joined = true;
        while (tc::ld_acquire_gpu_u32(cnt) < (uint32_t)S) {
          if (clock64() - t0 > p.wait_cycles) {
            *s_abort = 18;
            joined = false;
            break;
          }
        }
        __threadfence();
        // the last split past the barrier puts both counters back to zero for the next call
        // (every split has seen all arrivals before it counts its departure)
        if (joined && atomicAdd(dep, 1u) == (uint32_t)(S - 1)) {
          atomicExch(cnt, 0u);
          atomicExch(dep, 0u);
        }
      }
      ok = ok && all_sync() && *s_abort == 0;
      if (ok) {
        // Each thread merges items of 8 output dims of one head: it loads the (m, l) of
        // every split for that head and the split partials of its 8 dims, up to kJoinBatch
        // splits at once (all in flight together), and keeps a running maximum across
        // batches.  No shared table and no further barrier: one L2 round trip per batch.
        constexpr int kOcts = kC / 8;
        constexpr int kJoinBatch = 16;
        const int n_items = kHG * kOcts;
        const int i0 = (int)((int64_t)W.sp * n_items / S), i1 = (int)((int64_t)(W.sp + 1) * n_items / S);
        const float2* ml_b = p.part_ml + W.bq * S * p.n_h + W.hg * kHG;
        const __nv_bfloat16* po_b = p.part_o + (W.bq * S * p.n_hg + W.hg) * (int64_t)(kHG * kC);
        const int64_t split_stride = (int64_t)p.n_hg * kHG * kC;
        const int64_t o_b = (W.bq * p.n_h + W.hg * kHG) * kC;  // the unit's first output row
        for (int it = i0 + ts; it < i1; it += kSoftThreads) {
          const int h = it / kOcts, d = (it - h * kOcts) * 8;
          const int off = ((d >> 7) * kHG + h) * 128 + (d & 127);  // chunk-major partial
          float M = -INFINITY, L = 0.f, acc[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) acc[x] = 0.f;
          for (int s0 = 0; s0 < S; s0 += kJoinBatch) {
            float2 ml[kJoinBatch];
            uint4 raw[kJoinBatch];
#pragma unroll
            for (int j = 0; j < kJoinBatch; ++j) {
              const bool in = s0 + j < S;
              ml[j] = in ? __ldcg(&ml_b[(int64_t)(s0 + j) * p.n_h + h]) : make_float2(-INFINITY, 0.f);
              raw[j] = in ? __ldcg(reinterpret_cast<const uint4*>(po_b + (s0 + j) * split_stride + off))
                          : make_uint4(0u, 0u, 0u, 0u);
            }
            float Mb = M;
#pragma unroll
            for (int j = 0; j < kJoinBatch; ++j) Mb = fmaxf(Mb, ml[j].x);
            if (Mb == -INFINITY) continue;
            const float r = M == -INFINITY ? 0.f : exp2f(M - Mb);  // rescale what earlier batches added
            L *= r;
#pragma unroll
            for (int x = 0; x < 8; ++x) acc[x] *= r;
#pragma unroll
            for (int j = 0; j < kJoinBatch; ++j) {
              if (ml[j].x == -INFINITY) continue;
              const float e = exp2f(ml[j].x - Mb);
              L = fmaf(ml[j].y, e, L);
              const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[x]));
                acc[2 * x] = fmaf(e, v.x, acc[2 * x]);
                acc[2 * x + 1] = fmaf(e, v.y, acc[2 * x + 1]);
              }
            }
            M = Mb;
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
          for (int x = 0; x < 8; ++x) acc[x] *= inv;
          if (d == 0) p.lse[W.bq * p.n_h + W.hg * kHG + h] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
          const int64_t at = o_b + (int64_t)h * kC + d;
          if (MODE != 2 && p.win && p.out_bf16) {  // fused window merge: the merged output
            uint32_t pk[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * x], acc[2 * x + 1]);
              pk[x] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + at) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          } else {
            float* dst = (MODE != 2 && p.win) ? static_cast<float*>(p.out) : p.o;
            *reinterpret_cast<float4*>(dst + at) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(dst + at + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
          }
        }
      }
    }
  }
  __syncwarp();  // every warp reaches the CTA barrier converged
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT | ((*s_abort & 0xFF) << 8));
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

int64_t atc_list_len_max(const AttendJob& j) {
  if (j.mode == 0) return j.list_len;
  if (j.mode == 1)
    return j.q_pos ? j.n_entries : std::min<int64_t>(visible_entries(j.q_pos0 + j.n_q - 1, j.m), j.n_entries);
  return j.n_win;
}

}  // namespace

bool attend_tc_supported(const AttendJob& j) {
  if (j.dtype != HYB_BF16 || j.c != kC || j.n_h < kHG || j.n_h % kHG != 0) return false;
  if (j.win) {
    // a fused window joins with the list's splits: every CTA of the launch must be
    // resident at once (at most one per SM), so there must be room for two per unit
    const int64_t units = j.batch * j.n_q * (j.n_h / kHG);
    if (j.mode == 2 || units * 2 > kNumSMs || reinterpret_cast<uintptr_t>(j.wk) % 16 != 0) return false;
    if (j.batch * j.w_stride >= (int64_t(1) << 31)) return false;
  }
  const uintptr_t al = reinterpret_cast<uintptr_t>(j.q) | reinterpret_cast<uintptr_t>(j.k) |
                       reinterpret_cast<uintptr_t>(j.v);
  if (al % 16 != 0) return false;
  if (j.batch * j.n_q * j.n_h >= (int64_t(1) << 31) || j.batch * j.kv_stride >= (int64_t(1) << 31)) return false;
  return true;
}

namespace {

struct AtcPlan {
  int n_split;
};

// Splits of each (query, head group) list: every split CTA writes its partial (O, m, l)
// and the splits of a unit join through L2 inside the kernel.  A launch with splits
// has at most one CTA per SM, so all its CTAs are resident at once; the split count
// is the largest that fits, then evened out (the same tiles per CTA, fewer CTAs).
AtcPlan atc_plan(const AttendJob& j) {
  if (j.mode == 2) {
    // Window merge of one tile whose keys are its values: S CTAs per (query, head group)
    // each compute the (cheap) softmax and write 512/S of the output dims, merged with
    // their slice of the compressed branch's output; nothing is exchanged.
    if (j.k != j.v || atc_list_len_max(j) > kTile) return {1};
    const int64_t units = j.batch * j.n_q * (j.n_h / kHG);
    for (int S = 4; S >= 2; S >>= 1)
      if (units * S <= kNumSMs) return {S};
    return {1};
  }
  const int64_t T = (atc_list_len_max(j) + kTile - 1) / kTile;
  const int64_t units = j.batch * j.n_q * (j.n_h / kHG);
  const int w = j.win ? 1 : 0;  // a fused window is one more split, the last
  int64_t s = kNumSMs / std::max<int64_t>(units, 1) - w;
  s = std::min<int64_t>(std::min<int64_t>(s, T), kMaxSplits - w);
  if (s <= 1) return {1 + w};
  const int64_t per = (T + s - 1) / s;  // tiles per split
  return {(int)((T + per - 1) / per) + w};
}

}  // namespace

int attend_tc_splits(const AttendJob& j) { return atc_plan(j).n_split; }

size_t attend_tc_workspace_bytes(const AttendJob& j) {
  const AtcPlan pl = atc_plan(j);
  if (j.mode == 2) return 0;
  if (pl.n_split <= 1) return kJoinRegionBytes;
  const size_t n = (size_t)(j.batch * j.n_q * pl.n_split * j.n_h);
  return kJoinRegionBytes + n * (size_t)kC * sizeof(__nv_bfloat16) + n * sizeof(float2) + 256;
}

cudaError_t launch_attend_tc(const AttendJob& j, void* ws, cudaStream_t s) {
  if (j.batch == 0 || j.n_q == 0 || j.n_h == 0) return cudaSuccess;
  AtcParams p{};
  p.idx = j.idx;
  p.k = static_cast<const __nv_bfloat16*>(j.k);
  p.v = static_cast<const __nv_bfloat16*>(j.v);
  p.o = j.o, p.lse = j.lse;
  p.o_in = j.o_in, p.lse_in = j.lse_in, p.out = j.out, p.lse_out = j.lse, p.out_bf16 = j.out_bf16;
  p.n_q = j.n_q, p.n_h = j.n_h, p.n_entries = j.n_entries, p.kv_stride = j.kv_stride, p.list_len = j.list_len;
  p.m = j.m, p.q_pos0 = j.q_pos0, p.kv_pos0 = j.kv_pos0, p.n_win = j.n_win;
  const AtcPlan pl = atc_plan(j);
  p.n_split = pl.n_split;
  p.n_hg = (int)(j.n_h / kHG);
  p.alias = j.k == j.v;
  p.scale_log2 = j.scale * kLog2e;
  p.dev_status = j.dev_status;
  p.wait_cycles = grid_wait_cycles();
  p.win = j.win;
  p.kw = static_cast<const __nv_bfloat16*>(j.wk);
  p.w_stride = j.w_stride, p.w_pos0 = j.w_pos0, p.wq_pos0 = j.wq_pos0;
  p.q_pos = j.q_pos, p.kv_pos0s = j.kv_pos0s, p.wq_pos = j.wq_pos, p.w_pos0s = j.w_pos0s;
  const int64_t rows = j.batch * j.n_q;
  if (p.n_split > 1 && j.mode != 2) {
    if (rows * p.n_hg > kMaxJoinUnits) return cudaErrorInvalidConfiguration;  // (the plan never does this)
    const size_t n = (size_t)(rows * p.n_split * j.n_h);
    p.join_cnt = static_cast<uint32_t*>(ws);
    p.part_o = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(ws) + kJoinRegionBytes);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + kJoinRegionBytes +
                                          n * (size_t)kC * sizeof(__nv_bfloat16));
  }
  const uint64_t kv_rows = (uint64_t)(j.batch * j.kv_stride);
  const uint32_t box_rows = kv_rows < (uint64_t)kTile ? (uint32_t)kv_rows : (uint32_t)kTile;
  CUtensorMap tm_q, tm_k, tm_v, tm_w;
  if (!encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.q, kC, (uint64_t)(rows * j.n_h), kC * 2, 64, kHG,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.k, kC, kv_rows, kC * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.v, kC, kv_rows, kC * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  tm_w = tm_k;  // (unused without a fused window)
  if (j.win) {
    const uint64_t w_rows = (uint64_t)(j.batch * j.w_stride);
    const uint32_t w_box = w_rows < (uint64_t)kTile ? (uint32_t)w_rows : (uint32_t)kTile;
    if (!encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.wk, kC, w_rows, kC * 2, 64, w_box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int64_t grid = rows * p.n_split * p.n_hg;
  if (grid >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  auto run = [&](auto kernel) {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (r != cudaSuccess) return r;
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), (size_t)kSmemBytes, s, tm_q, tm_k, tm_v, tm_w,
                      p);
  };
  switch (j.mode) {
    case 0:
      e = run(attend_tc_kernel<0>);
      break;
    case 1:
      e = run(attend_tc_kernel<1>);
      break;
    default:
      e = run(attend_tc_kernel<2>);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
