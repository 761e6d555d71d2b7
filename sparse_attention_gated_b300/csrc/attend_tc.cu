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
// Warp roles (256 threads, one CTA per SM):
//   warps 0-2  producers: the query group by TMA once; entry slabs by TMA when
//              a tile is 128 consecutive rows, otherwise (index lists, ragged
//              last tile) gathered with 16-byte cp.async into the same
//              swizzled layout, rows without an entry zero-filled; for the
//              window merge, the compressed-branch output by one bulk copy.
//   warp 3     TMEM owner and MMA issuer (one elected thread).
//   warps 4-7  softmax and epilogue: thread e owns TMEM lane e (entry e of a
//              tile, head-dim row e of an O^T chunk).
// Online softmax in base 2 with a lazy reference: the per-head reference
// m[h] only moves when some score exceeds it by more than 2^8, which a
// block-wide vote detects; only then are the tile maxima reduced across the
// 128 entry lanes and the O^T accumulator rescaled.  Per-thread partial
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

constexpr int kHG = 64;                 // query heads per CTA (MMA N)
constexpr int kC = 512;                 // head dim c
constexpr int kTile = 128;              // entries per tile
constexpr int kSlabs = kC / 64;         // column slabs of 64 dims (128 bytes) per row
constexpr int kSlabBytes = kTile * 128;  // 16 KiB
constexpr int kQSlabBytes = kHG * 128;   // 8 KiB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kSlabs * kQSlabBytes;
constexpr int kOffP = kOffKV + kSlabs * kSlabBytes;
constexpr int kOffRed = kOffP + kTile * kHG * 2;
// float scratch: red[4][64], m[2][64], alpha[64], coef[2][64]
constexpr int kRedFloats = 4 * 64 + 2 * 64 + 64 + 2 * 64;
constexpr int kOffVote = kOffRed + kRedFloats * 4;
constexpr int kOffBar = kOffVote + 8 * 4;
constexpr int kNumBars = 1 + 2 * kSlabs + 2 + 2 + 1 + 1 + 1 + 1 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O^T: chunk ch at columns 64ch .. 64ch+63
constexpr uint32_t kTmemS = 256;  // S^T: buffer b at columns 256+64b ..
constexpr float kTau = 8.0f;      // lazy-reference threshold (log2 units): p <= 2^8
constexpr int kProdWarps = 3, kMmaWarp = 3, kSoftWarp0 = 4, kNumWarps = 8;
constexpr int kThreads = kNumWarps * 32;

static_assert(kSmemBytes <= 232448, "shared memory budget");

struct AtcParams {
  const int32_t* idx;       // mode 0: [rows][list_len]
  const __nv_bfloat16* k;   // gather sources, [batch][kv_stride][c]
  const __nv_bfloat16* v;
  float* o;                 // modes 0/1, one split: [rows][n_h][c]
  float* lse;               // [rows][n_h]
  float* part_o;            // modes 0/1, several splits: [rows][n_split][n_h][c]
  float2* part_ml;          // [rows][n_split][n_h] (reference m in log2 units, denominator)
  const float* o_in;        // mode 2
  const float* lse_in;
  void* out;
  float* lse_out;
  int out_bf16;
  int64_t n_q, n_h, n_entries, kv_stride, list_len, m, q_pos0, kv_pos0, n_win;
  int n_split, n_hg, alias;
  float scale_log2;
  int32_t* dev_status;
};

struct AtcWork {
  int64_t bq, b, j, hg, sp;
  int64_t L;     // list length of this query
  int64_t row0;  // modes 1/2: global row of list position 0
  const int32_t* list;
  int64_t tb, te;  // this split's tiles
};

template <int MODE>
__device__ __forceinline__ AtcWork atc_work(const AtcParams& p) {
  AtcWork w;
  const int64_t id = blockIdx.x;
  w.hg = id % p.n_hg;
  w.sp = (id / p.n_hg) % p.n_split;
  w.bq = id / ((int64_t)p.n_hg * p.n_split);
  w.b = w.bq / p.n_q;
  w.j = w.bq % p.n_q;
  const int64_t t = p.q_pos0 + w.j;
  w.list = nullptr;
  w.row0 = 0;
  if constexpr (MODE == 0) {
    w.L = p.list_len;
    w.list = p.idx + w.bq * p.list_len;
  } else if constexpr (MODE == 1) {
    const int64_t v = visible_entries(t, p.m);
    w.L = v < p.n_entries ? v : p.n_entries;
    w.row0 = w.b * p.kv_stride;
  } else {
    w.L = t + 1 < p.n_win ? t + 1 : p.n_win;
    w.row0 = w.b * p.kv_stride + (t - w.L + 1 - p.kv_pos0);
  }
  const int64_t T = (w.L + kTile - 1) / kTile;
  w.tb = w.sp * T / p.n_split;
  w.te = (w.sp + 1) * T / p.n_split;
  return w;
}

// Global row of list position pos, or -1 when the position holds no entry.
template <int MODE>
__device__ __forceinline__ int64_t atc_row(const AtcParams& p, const AtcWork& w, int64_t pos, bool report) {
  if (pos >= w.L) return -1;
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
// order by one warp.
template <int MODE>
__device__ __forceinline__ int atc_gather_warp(int64_t g) {
  return MODE == 0 ? (int)(g % kProdWarps) : 0;
}

// Reduce 64 per-lane values (a: heads 0-31, b: heads 32-63) across the 32
// lanes of a warp by recursive halving: after the five exchange steps lane l
// holds the reduction for heads 2l and 2l+1.  62 shuffles instead of 320.
template <bool MAX>
__device__ __forceinline__ void transpose_reduce(float (&a)[32], float (&b)[32], int lane, float& r0, float& r1) {
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float send = up ? a[i] : b[i];
      const float keep = up ? b[i] : a[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < 2 * o; ++i) {
      const float lo = a[i], hi = a[i + 2 * o];
      const float send = up ? lo : hi;
      const float keep = up ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      a[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  r0 = a[0];
  r1 = a[1];
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, AtcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem + kOffQ;
  uint8_t* kv_s = smem + kOffKV;
  uint8_t* p_s = smem + kOffP;
  float* red = reinterpret_cast<float*>(smem + kOffRed);  // [4][64]
  float* m_s = red + 4 * 64;                                // [2][64]
  float* alpha_s = m_s + 2 * 64;                            // [64]
  float* coef_s = alpha_s + 64;                             // [2][64]
  volatile int* vote = reinterpret_cast<volatile int*>(smem + kOffVote);  // [2][4]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;
  uint64_t* kv_empty = kv_full + kSlabs;
  uint64_t* s_full = kv_empty + kSlabs;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* sm_sync = o_done + 1;
  uint64_t* fin = sm_sync + 1;
  uint64_t* oin_full = fin + 1;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AtcWork W = atc_work<MODE>(p);
  const int64_t ntiles = W.te - W.tb;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < kSlabs; ++s) tc::mbar_init(&kv_full[s], 1), tc::mbar_init(&kv_empty[s], 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&s_full[i], 1), tc::mbar_init(&s_empty[i], 4);
    tc::mbar_init(p_full, 4);
    tc::mbar_init(o_done, 1);
    tc::mbar_init(sm_sync, 128);
    tc::mbar_init(fin, 1);
    tc::mbar_init(oin_full, 1);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(s_tmem, kTmemCols);
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_q);
    if (MODE != 0) {
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp < kProdWarps) {
    // ================================================================ producers
    bool ok = true;
    int pend[2];
    int npend = 0;
    int64_t tma_u[kSlabs];  // last use count of each slot filled by TMA (for the drain on abort)
#pragma unroll
    for (int s = 0; s < kSlabs; ++s) tma_u[s] = -1;
    // make this warp's finished gathers visible to the MMA and signal them
    auto flush = [&]() {
      if (npend) {
        tc::cp_async_wait_all();
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int x = 0; x < npend; ++x) tc::mbar_arrive(&kv_full[pend[x]]);
        npend = 0;
      }
    };
    if (warp == 0 && ntiles > 0) {
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(q_full, kSlabs * kQSlabBytes);
        const int32_t qrow = (int32_t)(W.bq * p.n_h + W.hg * kHG);
        for (int s = 0; s < kSlabs; ++s) tc::tma_load_2d(q_s + s * kQSlabBytes, &tm_q, q_full, 64 * s, qrow);
      }
      __syncwarp();
    }
    const int64_t ngroups = 2 * ntiles;
    int64_t g = 0;  // slab sequence number
    for (int64_t G = 0; G < ngroups && ok; ++G) {
      bool is_v;
      const int64_t li = atc_group(G, ngroups, is_v);
      const int64_t i = W.tb + li;
      const bool tma_tile = MODE != 0 && (i + 1) * kTile <= W.L;
      int64_t rows[4];
      if (!tma_tile) {
#pragma unroll
        for (int r = 0; r < 4; ++r) rows[r] = atc_row<MODE>(p, W, i * kTile + lane + 32 * r, warp == 0 && !is_v);
      }
      const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
      const __nv_bfloat16* src = is_v ? p.v : p.k;
      const uint32_t par = (uint32_t)(G & 1) ^ 1u;  // wait for the release of the slot's previous use
      // a TMA group after gathered slabs (ragged tile K, then the full tile's V) must not
      // block on a slot while this warp still holds copies it has not signalled
      if (tma_tile && warp == 0) flush();
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
        } else if (atc_gather_warp<MODE>(g) == warp) {
          int okl = 1;
          if (lane == 0) okl = tc::mbar_try_wait(&kv_empty[s], par);
          if (!__shfl_sync(0xffffffffu, okl, 0)) {
            flush();  // never block on a slot while holding un-signalled copies
            if (lane == 0) okl = tc::mbar_wait(&kv_empty[s], par, s_abort, 2);
            ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
            if (!ok) break;
          }
          const uint32_t dbase = tc::smem_u32(dst);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int e = lane + 32 * r;
            const bool have = rows[r] >= 0;
            const __nv_bfloat16* rsrc = src + (have ? rows[r] : 0) * kC + s * 64;
            const uint32_t drow = dbase + (uint32_t)((e >> 3) * 1024 + (e & 7) * 128);
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16)
              tc::cp_async16(drow + (uint32_t)((c16 ^ (e & 7)) << 4), rsrc + c16 * 8, have ? 16u : 0u);
          }
          tc::cp_async_commit();
          pend[npend++] = s;
          if (npend == 2) {
            tc::cp_async_wait_group<1>();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&kv_full[pend[0]]);
            pend[0] = pend[1];
            npend = 1;
          }
        }
      }
    }
    flush();
    bool oin_issued = false;
    if constexpr (MODE == 2) {
      // the compressed-branch output of this query's heads, into the ring once the last products are done
      if (ok && warp == 0 && p.o_in != nullptr && ntiles > 0) {
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
      const int64_t ngroups = 2 * ntiles;
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
            tc::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_f16(dS, tc::desc_kmajor_sw128(kv_addr + s * kSlabBytes + 32 * kk),
                          tc::desc_kmajor_sw128(q_addr + s * kQSlabBytes + 32 * kk), idS, (s | kk) ? 1u : 0u);
            tc::mma_commit(&kv_empty[s]);  // the slot is free once these products are done
          }
          if (!ok) break;
          tc::mma_commit(&s_full[sb]);
        } else {
          if (!(ok = tc::mbar_wait(p_full, (uint32_t)(li & 1), s_abort, 6))) break;
          tc::tc_fence_after();
          for (int ch = 0; ch < 4; ++ch) {
            if (!(ok = tc::mbar_wait(&kv_full[2 * ch], par, s_abort, 7))) break;
            if (!(ok = tc::mbar_wait(&kv_full[2 * ch + 1], par, s_abort, 7))) break;
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
    const int q4 = warp & 3;            // TMEM lane quadrant of this warp
    const int e = q4 * 32 + lane;       // tile entry / O^T chunk row owned by this thread
    const int st = threadIdx.x - kSoftWarp0 * 32;  // 0..127
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    uint32_t sync_phase = 0;
    auto gsync = [&]() -> bool {
      tc::mbar_arrive(sm_sync);
      const bool r = tc::mbar_wait(sm_sync, sync_phase, s_abort, 9);
      sync_phase ^= 1u;
      return r;
    };
    float lp[64];
#pragma unroll
    for (int h = 0; h < 64; ++h) lp[h] = 0.f;
    int mcur = 0;
    if (st < 64) m_s[st] = -INFINITY, m_s[64 + st] = -INFINITY;
    bool ok = gsync();

    for (int64_t li = 0; li < ntiles && ok; ++li) {
      const int64_t i = W.tb + li;
      const int sb = (int)(li & 1);
      if (!(ok = tc::mbar_wait(&s_full[sb], (uint32_t)((li >> 1) & 1), s_abort, 8))) break;
      tc::tc_fence_after();
      const uint32_t sS = tmem + lane_base + kTmemS + (uint32_t)(sb * kHG);
      const bool valid = atc_row<MODE>(p, W, i * kTile + e, false) >= 0;
      float sa[32], sb2[32];
      auto load_scores = [&]() {
        tc::tmem_ld32(sS, sa);
        tc::tmem_ld32(sS + 32, sb2);
        tc::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          sa[h] = valid ? sa[h] * p.scale_log2 : -INFINITY;
          sb2[h] = valid ? sb2[h] * p.scale_log2 : -INFINITY;
        }
      };
      load_scores();
      const float* mref = m_s + mcur * 64;
      bool exceed = false;
#pragma unroll
      for (int h = 0; h < 32; ++h) exceed |= (sa[h] > mref[h] + kTau) | (sb2[h] > mref[32 + h] + kTau);
      const int any_w = __any_sync(0xffffffffu, exceed);
      if (lane == 0) vote[sb * 4 + q4] = any_w;
      if (!(ok = gsync())) break;
      const bool any = (vote[sb * 4 + 0] | vote[sb * 4 + 1] | vote[sb * 4 + 2] | vote[sb * 4 + 3]) != 0;
      bool odone = false;
      if (any) {
        // move the reference to the tile maximum of every head
        float r0, r1;
        transpose_reduce<true>(sa, sb2, lane, r0, r1);
        red[q4 * 64 + 2 * lane] = r0;
        red[q4 * 64 + 2 * lane + 1] = r1;
        if (!(ok = gsync())) break;
        if (st < 64) {
          const float mo = mref[st];
          const float mn = fmaxf(fmaxf(mo, fmaxf(red[st], red[64 + st])), fmaxf(red[128 + st], red[192 + st]));
          m_s[(mcur ^ 1) * 64 + st] = mn;
          alpha_s[st] = mn == -INFINITY ? 1.f : exp2f(mo - mn);
        }
        if (!(ok = gsync())) break;
        mcur ^= 1;
#pragma unroll
        for (int h = 0; h < 64; ++h) lp[h] *= alpha_s[h];
        if (li > 0) {
          // rescale O^T once the previous tile's products are complete
          if (!(ok = tc::mbar_wait(o_done, (uint32_t)((li - 1) & 1), s_abort, 10))) break;
          odone = true;
          tc::tc_fence_after();
#pragma unroll 1
          for (int x = 0; x < 8; ++x) {
            float v[32];
            const uint32_t ta = tmem + lane_base + kTmemO + (uint32_t)(x * 32);
            tc::tmem_ld32(ta, v);
            tc::tmem_ld_wait();
            const float* al = alpha_s + (x & 1) * 32;
#pragma unroll
            for (int y = 0; y < 32; ++y) v[y] *= al[y];
            tc::tmem_st32(ta, v);
          }
          tc::tmem_st_wait();
        }
        load_scores();  // the reduction consumed the registers
      }
      // probabilities of this entry for every head, as row e of P^T (bf16)
      const float* mr = m_s + mcur * 64;
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 32; h += 2) {
        const float p0 = sa[h] == -INFINITY ? 0.f : exp2f(sa[h] - mr[h]);
        const float p1 = sa[h + 1] == -INFINITY ? 0.f : exp2f(sa[h + 1] - mr[h + 1]);
        const float p2 = sb2[h] == -INFINITY ? 0.f : exp2f(sb2[h] - mr[32 + h]);
        const float p3 = sb2[h + 1] == -INFINITY ? 0.f : exp2f(sb2[h + 1] - mr[33 + h]);
        lp[h] += p0, lp[h + 1] += p1, lp[32 + h] += p2, lp[33 + h] += p3;
        pk[h / 2] = pack_bf16x2(p0, p1);
        pk[16 + h / 2] = pack_bf16x2(p2, p3);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&s_empty[sb]);
      if (li > 0 && !odone) {
        if (!(ok = tc::mbar_wait(o_done, (uint32_t)((li - 1) & 1), s_abort, 11))) break;
      }
      uint8_t* prow = p_s + (e >> 3) * 1024 + (e & 7) * 128;
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4*>(prow + ((c16 ^ (e & 7)) << 4)) =
            make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(p_full);
    }

    if (ok) {
      // denominators: reduce the per-entry partial sums of every head across the 128 lanes
      {
        float la[32], lb[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) la[h] = lp[h], lb[h] = lp[32 + h];
        float r0, r1;
        transpose_reduce<false>(la, lb, lane, r0, r1);
        red[q4 * 64 + 2 * lane] = r0;
        red[q4 * 64 + 2 * lane + 1] = r1;
      }
      ok = gsync();
    }
    if (ok) {
      if (st < 64) {
        const int64_t H = W.hg * kHG + st;
        const float l = (red[st] + red[64 + st]) + (red[128 + st] + red[192 + st]);
        const float mm = m_s[mcur * 64 + st];
        const float lse2 = l > 0.f ? mm + __log2f(l) : -INFINITY;  // log2 of the denominator
        if constexpr (MODE == 2) {
          const float lse_w = lse2 * kLn2;
          const float lse_c = p.lse_in ? p.lse_in[W.bq * p.n_h + H] : -INFINITY;
          const float M = fmaxf(lse_w, lse_c);
          float wc = 0.f, ww = 0.f, Lse = -INFINITY;
          if (M != -INFINITY) {
            const float ec = lse_c == -INFINITY ? 0.f : expf(lse_c - M);
            const float ew = lse_w == -INFINITY ? 0.f : expf(lse_w - M);
            const float den = ec + ew;
            wc = ec / den;
            ww = ew / (den * (l > 0.f ? l : 1.f));  // the accumulator is unnormalised
            Lse = M + logf(den);
          }
          coef_s[st] = ww;
          coef_s[64 + st] = wc;
          if (p.lse_out) p.lse_out[W.bq * p.n_h + H] = Lse;
        } else if (p.n_split > 1) {
          coef_s[st] = 1.f;
          p.part_ml[(W.bq * p.n_split + W.sp) * p.n_h + H] = make_float2(l > 0.f ? mm : -INFINITY, l);
        } else {
          coef_s[st] = l > 0.f ? 1.f / l : 0.f;
          p.lse[W.bq * p.n_h + H] = lse2 * kLn2;
        }
      }
      ok = gsync();
    }
    if (ok && ntiles > 0) {
      ok = tc::mbar_wait(o_done, (uint32_t)((ntiles - 1) & 1), s_abort, 12);
      tc::tc_fence_after();
    }
    if constexpr (MODE == 2) {
      if (ok && p.o_in != nullptr) ok = tc::mbar_wait(oin_full, 0, s_abort, 14);
    }
    if (ok) {
      // O^T (TMEM) -> global: for a fixed head the 32 lanes of a warp store 32 consecutive dims
      float* obase;
      if constexpr (MODE == 2)
        obase = nullptr;
      else
        obase = p.n_split > 1 ? p.part_o + ((W.bq * p.n_split + W.sp) * p.n_h + W.hg * kHG) * kC
                              : p.o + (W.bq * p.n_h + W.hg * kHG) * kC;
#pragma unroll 1
      for (int x = 0; x < 8; ++x) {
        const int ch = x >> 1, h0 = (x & 1) * 32;
        float v[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(x * 32), v);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) v[y] = 0.f;
        }
        const int64_t d = ch * 128 + e;
        if constexpr (MODE == 2) {
          const int64_t rb = (W.bq * p.n_h + W.hg * kHG + h0) * kC + d;
          const float* oin = reinterpret_cast<const float*>(kv_s) + h0 * kC + d;  // staged o_in, [64][512]
#pragma unroll
          for (int y = 0; y < 32; ++y) {
            const float wc = coef_s[64 + h0 + y];
            const float r = coef_s[h0 + y] * v[y] + (wc != 0.f ? wc * oin[y * kC] : 0.f);
            if (p.out_bf16)
              static_cast<__nv_bfloat16*>(p.out)[rb + (int64_t)y * kC] = __float2bfloat16_rn(r);
            else
              static_cast<float*>(p.out)[rb + (int64_t)y * kC] = r;
          }
        } else {
#pragma unroll
          for (int y = 0; y < 32; ++y) obase[(int64_t)(h0 + y) * kC + d] = v[y] * coef_s[h0 + y];
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT | ((*s_abort & 0xFF) << 8));
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the split partials of every (query, head): one CTA of 128 threads per
// (query, head), four dims per thread.
__global__ void __launch_bounds__(128) atc_combine_kernel(const float* __restrict__ part_o,
                                                          const float2* __restrict__ part_ml, float* o, float* lse,
                                                          int64_t n_h, int n_split) {
  const int64_t bq = blockIdx.x / n_h, h = blockIdx.x % n_h;
  const int d = threadIdx.x * 4;
  float M = -INFINITY;
  for (int sp = 0; sp < n_split; ++sp) M = fmaxf(M, part_ml[(bq * n_split + sp) * n_h + h].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  if (M != -INFINITY) {
#pragma unroll 8
    for (int sp = 0; sp < n_split; ++sp) {
      const int64_t pi = (bq * n_split + sp) * n_h + h;
      const float2 ml = part_ml[pi];
      const float wgt = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
      l = fmaf(wgt, ml.y, l);
      const float4 po = __ldg(reinterpret_cast<const float4*>(part_o + pi * kC + d));
      acc.x = fmaf(wgt, po.x, acc.x);
      acc.y = fmaf(wgt, po.y, acc.y);
      acc.z = fmaf(wgt, po.z, acc.z);
      acc.w = fmaf(wgt, po.w, acc.w);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  acc.x *= inv, acc.y *= inv, acc.z *= inv, acc.w *= inv;
  *reinterpret_cast<float4*>(o + (bq * n_h + h) * kC + d) = acc;
  if (threadIdx.x == 0) lse[bq * n_h + h] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
}

int64_t atc_list_len_max(const AttendJob& j) {
  if (j.mode == 0) return j.list_len;
  if (j.mode == 1) return std::min<int64_t>(visible_entries(j.q_pos0 + j.n_q - 1, j.m), j.n_entries);
  return j.n_win;
}

}  // namespace

bool attend_tc_supported(const AttendJob& j) {
  if (j.dtype != HYB_BF16 || j.c != kC || j.n_h < kHG || j.n_h % kHG != 0) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(j.q) | reinterpret_cast<uintptr_t>(j.k) |
                       reinterpret_cast<uintptr_t>(j.v);
  if (al % 16 != 0) return false;
  if (j.batch * j.n_q * j.n_h >= (int64_t(1) << 31) || j.batch * j.kv_stride >= (int64_t(1) << 31)) return false;
  return true;
}

int attend_tc_splits(const AttendJob& j) {
  if (j.mode == 2) return 1;
  const int64_t T = (atc_list_len_max(j) + kTile - 1) / kTile;
  const int64_t units = j.batch * j.n_q * (j.n_h / kHG);
  int64_t s = kNumSMs / std::max<int64_t>(units, 1);
  s = std::min<int64_t>(s, T);
  s = std::min<int64_t>(s, 64);
  return (int)std::max<int64_t>(s, 1);
}

size_t attend_tc_workspace_bytes(const AttendJob& j) {
  const int s = attend_tc_splits(j);
  if (s <= 1) return 0;
  const size_t n = (size_t)(j.batch * j.n_q * s * j.n_h);
  return n * (size_t)kC * sizeof(float) + n * sizeof(float2) + 256;
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
  p.n_split = attend_tc_splits(j);
  p.n_hg = (int)(j.n_h / kHG);
  p.alias = j.k == j.v;
  p.scale_log2 = j.scale * kLog2e;
  p.dev_status = j.dev_status;
  const int64_t rows = j.batch * j.n_q;
  if (p.n_split > 1) {
    const size_t n = (size_t)(rows * p.n_split * j.n_h);
    p.part_o = static_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws) + n * (size_t)kC * sizeof(float));
  }
  const uint64_t kv_rows = (uint64_t)(j.batch * j.kv_stride);
  const uint32_t box_rows = kv_rows < (uint64_t)kTile ? (uint32_t)kv_rows : (uint32_t)kTile;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.q, kC, (uint64_t)(rows * j.n_h), kC * 2, 64, kHG,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.k, kC, kv_rows, kC * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, j.v, kC, kv_rows, kC * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t grid = rows * p.n_split * p.n_hg;
  if (grid >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  switch (j.mode) {
    case 0:
      e = cudaFuncSetAttribute(attend_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e == cudaSuccess) attend_tc_kernel<0><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(tm_q, tm_k, tm_v, p);
      break;
    case 1:
      e = cudaFuncSetAttribute(attend_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e == cudaSuccess) attend_tc_kernel<1><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(tm_q, tm_k, tm_v, p);
      break;
    default:
      e = cudaFuncSetAttribute(attend_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e == cudaSuccess) attend_tc_kernel<2><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(tm_q, tm_k, tm_v, p);
      break;
  }
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_split > 1) {
    atc_combine_kernel<<<(unsigned)(rows * j.n_h), 128, 0, s>>>(p.part_o, p.part_ml, j.o, j.lse, j.n_h, p.n_split);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace hyb
