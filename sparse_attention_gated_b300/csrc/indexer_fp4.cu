// indexer_fp4.cu -- lightning-indexer scores with MXFP4 queries and keys on the tensor cores
// ("DeepSeek-V4 hybrid attention" (trishampatil.com) section V.2 for the score; "DeepSeek-V4:
// Anatomy of an Open-Source Frontier Model" (modernaiengineering.com), "FP4 quantization-aware
// training": V4 runs the indexer's query-key path in FP4).
//
//   I[t,s] = sum_h w[t,h] * ReLU( sum_blk 2^(eq[t,h,blk] + ek[s,blk] - 254) * sum_{i in blk} q_i k_i )
//
// where q_i, k_i are e2m1 values and eq, ek the e8m0 scale bytes of their block of 32 dims.
// The keys stay packed in HBM (64 bytes + 4 scale bytes per entry, against 132 for FP8).  On
// chip every e2m1 value is written as an e4m3 byte, and the products run as tcgen05.mma
// kind::f8f6f4 (M = 128 entries, N = 64 heads, K = 32 per block), in one of two ways per tile:
//   folded  (every key row of the tile and every head of the query has block exponents within
//           8 of its largest, R): each value is written as the e4m3 byte of value * 2^(e - R),
//           exact (e2m1's magnitudes 0.5 .. 6 times 2^0 .. 2^-8 are all e4m3 numbers), the four
//           blocks accumulate into one TMEM accumulator, and the epilogue applies 2^(Rk + Rq
//           - 254) per (entry, head), as the FP8 path applies its row scales;
//   blocked (otherwise): each value is written as the e4m3 byte of the same value, each block
//           is one product into its own accumulator, and the epilogue combines the four with
//           their two scales.
//
// Roles (one CTA of 448 threads per SM, persistent over units = (query row, run of tiles)):
//   warp 0      TMA producer: the unit's packed query rows, then per tile of 128 entries the
//               packed keys (8 KiB) and their scale words (512 B) into a ring;
//   warp 1      TMEM owner and MMA issuer;
//   warps 2-5   expand packed tiles into e4m3 tiles (128-byte swizzle) for the MMA, 32 rows
//               per warp, and the unit's query rows, and hand the scale words to the epilogue;
//   warps 6-13  epilogue in two groups of four taking alternate tiles: an entry row's
//               products, the scales, ReLU and the head weights, one float32 score per
//               (query, entry), and (decode) the row's 12-bit score-key histogram.
// Accumulators: 8 slots of 64 TMEM columns (tile i in slot i % 8), so that the MMA runs up to
// 8 tiles ahead of the epilogue; a folded tile takes one turn of its slot, a blocked tile four
// (block k's product, read and released by the epilogue before block k + 1's is issued).
// Every wait is bounded (about 1 s): on expiry HYB_DEV_TIMEOUT is raised, the CTA's own copies
// and products in flight land, TMEM is freed and the kernel returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace hyb {

namespace {

constexpr int kTileE = 128;                 // entries per tile (MMA M)
constexpr int kHeads = 64;                  // indexer heads (MMA N)
constexpr int kRowRaw = 64;                 // packed bytes per 128-dim row
constexpr int kRawKeyBytes = kTileE * kRowRaw;    // 8 KiB
constexpr int kRawScaleBytes = kTileE * 4;        // one 4-byte word (4 e8m0 bytes) per entry
constexpr int kF8Bytes = kTileE * 128;            // 16 KiB: e4m3, 128-byte swizzle
constexpr int kRawQBytes = kHeads * kRowRaw;      // 4 KiB
constexpr int kQ8Bytes = kHeads * 128;            // 8 KiB
constexpr int kSR = 8;                      // packed-tile ring
constexpr int kS8 = 4;                      // e4m3 tile ring
constexpr int kAcc = 8;                     // accumulator slots of 64 columns
constexpr int kScaleRing = kS8 + kAcc;      // scale words on their way to the epilogue
constexpr int kThreads = 448;               // 14 warps: 4 on the busiest scheduler, so <= 128 registers each
constexpr int kConvWarp0 = 2, kConvGroups = 1;
constexpr int kConv = 4;                    // converter warps per group (one tile's arrivals)
constexpr int kEpiWarp0 = kConvWarp0 + kConvGroups * kConv, kEpiWarps = 8, kEpiGroups = 2;
static_assert((kEpiWarp0 + kEpiWarps) * 32 == kThreads, "warp roles");
constexpr int kEpiThreads = kEpiWarps * 32;

constexpr int kOffF8 = 0;
constexpr int kOffQ8 = kOffF8 + kS8 * kF8Bytes;
constexpr int kOffRaw = kOffQ8 + 2 * kQ8Bytes;
constexpr int kOffRawS = kOffRaw + kSR * kRawKeyBytes;
constexpr int kOffRawQ = kOffRawS + kSR * kRawScaleBytes;
constexpr int kOffQ8f = kOffRawQ + 2 * kRawQBytes;            // the folded query tiles
constexpr int kOffKS = kOffQ8f + 2 * kQ8Bytes;
constexpr int kOffQS = kOffKS + kScaleRing * kRawScaleBytes;  // float [64][4] query block scales, [64] 2^(Rq-127), w [64]
constexpr int kOffFlag = kOffQS + kHeads * 6 * 4;             // per scale slot: 1 = the tile is folded
constexpr int kOffTab = kOffFlag + kScaleRing * 4;            // uint32 [9][2]: e4m3 bytes of e2m1 magnitudes * 2^-d
constexpr int kOffHist = (kOffTab + 9 * 2 * 4 + 15) / 16 * 16;  // 16-bit counters, two per word (read as uint4)
constexpr int kOffBar = kOffHist + kTopkHistBins * 2;
static_assert(kOffF8 % 1024 == 0 && kOffQ8 % 1024 == 0 && kOffQ8f % 1024 == 0, "128-byte swizzled tiles");
static_assert(kOffRaw % 128 == 0 && kOffRawS % 128 == 0 && kOffRawQ % 128 == 0, "TMA destinations");
static_assert(kOffKS % 16 == 0 && kOffQS % 16 == 0 && kOffHist % 16 == 0 && kOffBar % 8 == 0, "vector and mbarrier alignment");
enum {
  kBarRawFull = 0,
  kBarRawEmpty = kBarRawFull + kSR,
  kBarF8Full = kBarRawEmpty + kSR,
  kBarF8Empty = kBarF8Full + kS8,
  kBarRqFull = kBarF8Empty + kS8,
  kBarRqEmpty = kBarRqFull + 2,
  kBarQ8Full = kBarRqEmpty + 2,
  kBarQ8Empty = kBarQ8Full + 2,
  kBarAccFull = kBarQ8Empty + 2,
  kBarAccEmpty = kBarAccFull + kAcc,
  kBarKsFull = kBarAccEmpty + kAcc,
  kBarKsEmpty = kBarKsFull + kScaleRing,
  kBarDone = kBarKsEmpty + kScaleRing,
  kBarEpi = kBarDone + 1,
  kNumBars = kBarEpi + 1
};
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + flags + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kTopkHistBins % 16 == 0, "the histogram in 8-word slices");

struct Fp4Params {
  const float* w;
  const uint8_t* qI_scale;  // [rows][64][4] e8m0
  float* scores;
  uint32_t* ghist;
  int64_t score_stride;
  int64_t n_q, n_entries, kv_stride, m, q_pos0;
  const int64_t* q_pos;
  int64_t tiles_per_unit, units_per_group, n_units;
  int32_t* dev_status;
};

struct Fp4Unit {
  int64_t b, j, row, tile_begin, tile_end;
};

__device__ __forceinline__ Fp4Unit fp4_unit(const Fp4Params& p, int64_t u) {
  Fp4Unit U;
  const int64_t g = u / p.units_per_group, chunk = u % p.units_per_group;
  U.row = g, U.b = g / p.n_q, U.j = g % p.n_q;
  const int64_t vis = visible_checked(query_pos(p.q_pos, p.q_pos0, U.row, U.j), p.m, p.n_entries, nullptr, false);
  const int64_t tiles = (vis + kTileE - 1) / kTileE;
  U.tile_begin = chunk * p.tiles_per_unit;
  U.tile_end = U.tile_begin + p.tiles_per_unit < tiles ? U.tile_begin + p.tiles_per_unit : tiles;
  return U;
}

// 2^(e - 127) for an e8m0 byte (255 is NaN), as a float32
__device__ __forceinline__ float e8m0_value(uint32_t e) {
  return e == 255u ? __uint_as_float(0x7FC00000u) : e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// e4m3 byte of the e2m1 code v (bit 3 the sign): 0, 0.5, 1, 1.5, 2, 3, 4, 6 exactly
__host__ __device__ constexpr uint32_t e2m1_to_e4m3(uint32_t v) {
  constexpr uint8_t mag[8] = {0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C};
  return (uint32_t)mag[v & 7u] | ((v & 8u) << 4);
}

// e4m3 byte of the e2m1 magnitude m (0..7) times 2^-d, d in 0..8: exact.  The magnitudes
// are 1.0 or 1.5 times 2^-1 .. 2^2; scaled, a normal e4m3 number has exponent field E + 7 >= 1,
// below that the subnormal (field 0) holds (2 + half) * 2^(E + 8) units of 2^-9.
__host__ __device__ constexpr uint32_t e4m3_of_e2m1(uint32_t m, int d) {
  constexpr int em[8] = {0, -1, 0, 0, 1, 1, 2, 2};
  constexpr int hf[8] = {0, 0, 0, 1, 0, 1, 0, 1};
  if (m == 0) return 0u;
  const int E = em[m] - d, h = hf[m];
  if (E >= -6) return (uint32_t)(((E + 7) << 3) | (h << 2));
  return E == -9 ? 1u : (uint32_t)((2 + h) << (E + 8));
}
__host__ __device__ constexpr uint32_t mag_table(int d, int half) {
  return e4m3_of_e2m1(4 * half, d) | (e4m3_of_e2m1(4 * half + 1, d) << 8) | (e4m3_of_e2m1(4 * half + 2, d) << 16) |
         (e4m3_of_e2m1(4 * half + 3, d) << 24);
}
static_assert(mag_table(0, 0) == (e2m1_to_e4m3(0) | (e2m1_to_e4m3(1) << 8) | (e2m1_to_e4m3(2) << 16) |
                                  (e2m1_to_e4m3(3) << 24)), "unscaled table");

// e4m3 bytes of four packed e2m1 codes (the 16 low bits of v, element i in nibble i): the
// nibbles' magnitudes select from the byte tables lo/hi (one byte permute), their signs
// select 0x00 or 0x80 (another).
__device__ __forceinline__ uint32_t expand4(uint32_t v, uint32_t lo, uint32_t hi) {
  return __byte_perm(lo, hi, v & 0x7777u) | __byte_perm(0x00008000u, 0u, (v >> 3) & 0x1111u);
}

// Largest and smallest of a word's four e8m0 bytes
__device__ __forceinline__ void exp_range(uint32_t w4, uint32_t& mx, uint32_t& mn) {
  const uint32_t b0 = w4 & 0xFFu, b1 = (w4 >> 8) & 0xFFu, b2 = (w4 >> 16) & 0xFFu, b3 = w4 >> 24;
  mx = max(max(b0, b1), max(b2, b3));
  mn = min(min(b0, b1), min(b2, b3));
}

__global__ void __launch_bounds__(kThreads, 1)
    index_fp4_kernel(const __grid_constant__ CUtensorMap tm_keys, const __grid_constant__ CUtensorMap tm_ks,
                     const __grid_constant__ CUtensorMap tm_q, Fp4Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* f8 = smem + kOffF8;
  uint8_t* q8 = smem + kOffQ8;
  uint8_t* raw = smem + kOffRaw;
  uint32_t* raw_s = reinterpret_cast<uint32_t*>(smem + kOffRawS);
  uint8_t* raw_q = smem + kOffRawQ;
  uint8_t* q8f = smem + kOffQ8f;
  uint32_t* ks_ring = reinterpret_cast<uint32_t*>(smem + kOffKS);
  float* qs_t = reinterpret_cast<float*>(smem + kOffQS);  // [64][4]
  float* wq_t = qs_t + kHeads * 4;                         // [64]: w[h] * 2^(Rq[h] - 127)
  float* w_t = wq_t + kHeads;                              // [64]
  volatile int* tile_fast = reinterpret_cast<volatile int*>(smem + kOffFlag);
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + kOffTab);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + kNumBars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kNumBars) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSR; ++i) tc::mbar_init(&bars[kBarRawFull + i], 1), tc::mbar_init(&bars[kBarRawEmpty + i], kConv);
    for (int i = 0; i < kS8; ++i) tc::mbar_init(&bars[kBarF8Full + i], kConv), tc::mbar_init(&bars[kBarF8Empty + i], 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars[kBarRqFull + i], 1), tc::mbar_init(&bars[kBarRqEmpty + i], kConv);
      tc::mbar_init(&bars[kBarQ8Full + i], kConv), tc::mbar_init(&bars[kBarQ8Empty + i], 1);
    }
    for (int i = 0; i < kAcc; ++i)
      tc::mbar_init(&bars[kBarAccFull + i], 1), tc::mbar_init(&bars[kBarAccEmpty + i], kEpiWarps / kEpiGroups);
    for (int i = 0; i < kScaleRing; ++i)
      tc::mbar_init(&bars[kBarKsFull + i], kConv), tc::mbar_init(&bars[kBarKsEmpty + i], kEpiWarps / kEpiGroups);
    tc::mbar_init(&bars[kBarDone], 1);
    tc::mbar_init(&bars[kBarEpi], kEpiThreads);
    *s_abort = 0;
    tc::fence_barrier_init();
  }
  if (threadIdx.x < 18) tab[threadIdx.x] = mag_table(threadIdx.x >> 1, threadIdx.x & 1);
  if (warp == 1) tc::tmem_alloc(s_tmem, 512);
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_keys);
    tc::prefetch_tmap(&tm_ks);
    tc::prefetch_tmap(&tm_q);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // (the setup above touched only shared memory, TMEM and the parameters)
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t seq = 0, qc = 0, issued = 0;
      bool ok = true;
      int64_t q_last[2] = {-1, -1};  // last query load issued into each buffer (drained on abort)
      for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        const Fp4Unit U = fp4_unit(p, u);
        if (U.tile_begin >= U.tile_end) continue;
        const int qb = (int)(qc & 1);
        if (!(ok = tc::mbar_wait(&bars[kBarRqEmpty + qb], (uint32_t)((qc >> 1) & 1) ^ 1u, s_abort, 1))) break;
        tc::mbar_arrive_expect_tx(&bars[kBarRqFull + qb], kRawQBytes);
        tc::tma_load_2d(raw_q + qb * kRawQBytes, &tm_q, &bars[kBarRqFull + qb], 0, (int32_t)(U.row * kHeads));
        q_last[qb] = qc;
        ++qc;
        for (int64_t t = U.tile_begin; t < U.tile_end; ++t, ++seq) {
          const int rs = (int)(seq % kSR);
          if (!(ok = tc::mbar_wait(&bars[kBarRawEmpty + rs], (uint32_t)((seq / kSR) & 1) ^ 1u, s_abort, 2))) break;
          tc::mbar_arrive_expect_tx(&bars[kBarRawFull + rs], kRawKeyBytes + kRawScaleBytes);
          tc::tma_load_2d(raw + rs * kRawKeyBytes, &tm_keys, &bars[kBarRawFull + rs], 0,
                          (int32_t)(U.b * p.kv_stride + t * kTileE));
          tc::tma_load_2d(raw_s + rs * kTileE, &tm_ks, &bars[kBarRawFull + rs], (int32_t)(t * kTileE), (int32_t)U.b);
          ++issued;
        }
      }
      if (!ok) {
        // let this thread's copies in flight land before the CTA can exit
        for (int64_t i = issued > kSR ? issued - kSR : 0; i < issued; ++i)
          tc::mbar_wait_drain(&bars[kBarRawFull + i % kSR], (uint32_t)((i / kSR) & 1));
        for (int b = 0; b < 2; ++b)
          if (q_last[b] >= 0) tc::mbar_wait_drain(&bars[kBarRqFull + b], (uint32_t)((q_last[b] >> 1) & 1));
      }
    }
    __syncwarp();
  } else if (warp >= kConvWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------ expand packed -> e4m3
    // kConvGroups groups of 128 threads, group g taking the tiles with seq % kConvGroups == g;
    // thread x of a group takes row x of a key tile (group 0, of the unit's query tile: rows x of the plain
    // copy for x < 64, rows x - 64 of the folded copy otherwise): the row's 64 packed bytes
    // become its 128 e4m3 bytes, 16-byte chunk c of the row written at chunk c ^ (row & 7)
    // (128-byte swizzle), each 32-dim block with its table.
    const int cgrp = (warp - kConvWarp0) / kConv, cw = (warp - kConvWarp0) % kConv;
    const int x = cw * 32 + lane;
    // one row: tables lo/hi per block (d = the block's distance below the row's largest
    // exponent when folded, 0 otherwise)
    auto convert_row = [&](const uint8_t* src, uint8_t* dst, int row, uint32_t w4, bool fold) {
      uint32_t lo[4], hi[4];
      uint32_t mx = 0, mn = 0;
      if (fold) exp_range(w4, mx, mn);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int d = fold ? (int)(mx - ((w4 >> (8 * b)) & 0xFFu)) : 0;
        lo[b] = tab[2 * d], hi[b] = tab[2 * d + 1];
      }
      const uint4* s4 = reinterpret_cast<const uint4*>(src + row * kRowRaw);
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16 packed bytes = 32 values = block q = output chunks 2q, 2q + 1
        const uint4 v = s4[q];
        const uint4 o0 = make_uint4(expand4(v.x, lo[q], hi[q]), expand4(v.x >> 16, lo[q], hi[q]),
                                    expand4(v.y, lo[q], hi[q]), expand4(v.y >> 16, lo[q], hi[q]));
        const uint4 o1 = make_uint4(expand4(v.z, lo[q], hi[q]), expand4(v.z >> 16, lo[q], hi[q]),
                                    expand4(v.w, lo[q], hi[q]), expand4(v.w >> 16, lo[q], hi[q]));
        *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * q) ^ (row & 7)) << 4)) = o0;
        *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * q + 1) ^ (row & 7)) << 4)) = o1;
      }
    };
    int64_t seq = 0, qc = 0;
    bool ok = true;
    auto done = [&](uint64_t* bar) {
      tc::fence_proxy_async_smem();  // the e4m3 tiles are read by the tensor cores
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar);
    };
    for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
      const Fp4Unit U = fp4_unit(p, u);
      if (U.tile_begin >= U.tile_end) continue;
      const int qb = (int)(qc & 1);
      const uint32_t qpar = (uint32_t)((qc >> 1) & 1);
      int okw = 1;
      if (lane == 0 && cgrp == 0)
        okw = tc::mbar_wait(&bars[kBarRqFull + qb], qpar, s_abort, 3) &&
              tc::mbar_wait(&bars[kBarQ8Empty + qb], qpar ^ 1u, s_abort, 4);
      if (!(ok = __shfl_sync(0xffffffffu, okw, 0) != 0)) break;
      // the query heads' block exponents (each warp reads all 64 heads: both decide alike)
      const uint32_t* qsw = reinterpret_cast<const uint32_t*>(p.qI_scale) + U.row * kHeads;
      const uint32_t qw0 = __ldg(qsw + lane), qw1 = __ldg(qsw + 32 + lane);
      uint32_t qmx0, qmn0, qmx1, qmn1;
      exp_range(qw0, qmx0, qmn0);
      exp_range(qw1, qmx1, qmn1);
      const bool unit_fold = __all_sync(0xffffffffu, qmx0 - qmn0 <= 8u && qmx1 - qmn1 <= 8u);
      if (cgrp == 0) {
        // head x & 63: its scale word is this lane's qw0 (heads 0-31) or qw1 (heads 32-63)
        const uint32_t w4 = (cw & 1) ? qw1 : qw0;
        if (cw < 2)
          convert_row(raw_q + qb * kRawQBytes, q8 + qb * kQ8Bytes, x, w4, false);
        else if (unit_fold)
          convert_row(raw_q + qb * kRawQBytes, q8f + qb * kQ8Bytes, x - 64, w4, true);
        done(&bars[kBarQ8Full + qb]);
        if (lane == 0) tc::mbar_arrive(&bars[kBarRqEmpty + qb]);
      }
      ++qc;
      for (int64_t t = U.tile_begin; t < U.tile_end && ok; ++t, ++seq) {
        if ((int)(seq % kConvGroups) != cgrp) continue;  // the other group's tile
        const int rs = (int)(seq % kSR), s8 = (int)(seq % kS8), r = (int)(seq % kScaleRing);
        okw = 1;
        if (lane == 0)
          okw = tc::mbar_wait(&bars[kBarRawFull + rs], (uint32_t)((seq / kSR) & 1), s_abort, 5) &&
                tc::mbar_wait(&bars[kBarF8Empty + s8], (uint32_t)((seq / kS8) & 1) ^ 1u, s_abort, 6) &&
                tc::mbar_wait(&bars[kBarKsEmpty + r], (uint32_t)((seq / kScaleRing) & 1) ^ 1u, s_abort, 7);
        if (!(ok = __shfl_sync(0xffffffffu, okw, 0) != 0)) break;
        const uint8_t* src = raw + rs * kRawKeyBytes;
        const uint32_t* sw = raw_s + rs * kTileE;
        uint8_t* dst = f8 + s8 * kF8Bytes;
        // folded when every key row of the tile (each warp checks all 128) and the query allow it
        bool fold = unit_fold;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t mx, mn;
          exp_range(sw[32 * i + lane], mx, mn);
          fold = fold && mx - mn <= 8u;
        }
        fold = __all_sync(0xffffffffu, fold);
        convert_row(src, dst, x, sw[x], fold);
        if (x == 0) tile_fast[r] = fold ? 1 : 0;
        ks_ring[r * kTileE + x] = sw[x];
        done(&bars[kBarF8Full + s8]);
        if (lane == 0) {
          tc::mbar_arrive(&bars[kBarKsFull + r]);
          tc::mbar_arrive(&bars[kBarRawEmpty + rs]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (tc::elect_one()) {
      constexpr uint32_t idesc = tc::make_idesc(0, 0, 0, 0, kTileE, kHeads);  // e4m3 x e4m3, both K-major
      int64_t seq = 0, qc = 0;
      uint32_t tpar = 0;  // bit a: parity of slot a's completed turns (a register, not an indexed array)
      bool ok = true;
      for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        const Fp4Unit U = fp4_unit(p, u);
        if (U.tile_begin >= U.tile_end) continue;
        const int qb = (int)(qc & 1);
        if (!(ok = tc::mbar_wait(&bars[kBarQ8Full + qb], (uint32_t)((qc >> 1) & 1), s_abort, 8))) break;
        const uint32_t b_plain = tc::smem_u32(q8 + qb * kQ8Bytes), b_fold = tc::smem_u32(q8f + qb * kQ8Bytes);
        for (int64_t t = U.tile_begin; t < U.tile_end && ok; ++t, ++seq) {
          const int s8 = (int)(seq % kS8), a = (int)(seq % kAcc);
          const uint32_t d = tmem + (uint32_t)(a * kHeads);
          if (!(ok = tc::mbar_wait(&bars[kBarF8Full + s8], (uint32_t)((seq / kS8) & 1), s_abort, 10))) break;
          const uint32_t a_base = tc::smem_u32(f8 + s8 * kF8Bytes);
          if (tile_fast[seq % kScaleRing]) {
            // folded: the four blocks into one accumulator, one turn of the slot
            if (!(ok = tc::mbar_wait(&bars[kBarAccEmpty + a], ((tpar >> a) & 1u) ^ 1u, s_abort, 9))) break;
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_f8f6f4(d, tc::desc_kmajor_sw128(a_base + 32 * k), tc::desc_kmajor_sw128(b_fold + 32 * k), idesc,
                             k > 0 ? 1u : 0u);
            tc::mma_commit(&bars[kBarAccFull + a]);
            tpar ^= 1u << a;
          } else {
            // blocked: block k (dims 32k .. 32k+31) alone, one turn of the slot each
            for (int k = 0; k < 4 && ok; ++k) {
              if (!(ok = tc::mbar_wait(&bars[kBarAccEmpty + a], ((tpar >> a) & 1u) ^ 1u, s_abort, 9))) break;
              tc::tc_fence_after();
              tc::mma_f8f6f4(d, tc::desc_kmajor_sw128(a_base + 32 * k), tc::desc_kmajor_sw128(b_plain + 32 * k), idesc,
                             0u);
              tc::mma_commit(&bars[kBarAccFull + a]);
              tpar ^= 1u << a;
            }
            if (!ok) break;
          }
          tc::mma_commit(&bars[kBarF8Empty + s8]);
        }
        if (!ok) break;
        tc::mma_commit(&bars[kBarQ8Empty + qb]);
        ++qc;
      }
      tc::mma_commit(&bars[kBarDone]);  // completes once, after every product above
      tc::mbar_wait_drain(&bars[kBarDone], 0);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const int quad = warp & 3;
    const int grp = (warp - kEpiWarp0) / 4;  // tiles with seq % kEpiGroups == grp
    uint32_t ephase = 0;
    auto esync = [&]() -> bool {
      tc::mbar_arrive(&bars[kBarEpi]);
      const bool r = tc::mbar_wait(&bars[kBarEpi], ephase, s_abort, 11);
      ephase ^= 1u;
      return r;
    };
    const bool do_hist = p.ghist != nullptr;
    int64_t hist_row = -1;
    if (do_hist)
      for (int i = et; i < kTopkHistBins / 2; i += kEpiThreads) hist[i] = 0;
    auto flush_hist = [&](bool clear) {
      for (int sl = et; sl < kTopkHistBins / 16; sl += kEpiThreads) {  // slice sl: bins 16 sl .. 16 sl + 15
        uint4* h4 = reinterpret_cast<uint4*>(hist) + 2 * sl;
        const uint4 a = h4[0], b = h4[1];
        const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t* g = p.ghist + hist_row * kTopkHistBins + 16 * sl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (v[i] & 0xFFFFu) atomicAdd(g + 2 * i, v[i] & 0xFFFFu);
          if (v[i] >> 16) atomicAdd(g + 2 * i + 1, v[i] >> 16);
        }
        if (clear) h4[0] = h4[1] = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    int64_t seq = 0;
    uint32_t tpar = 0;  // bit a: parity of slot a's completed turns (this group's slots only)
    bool ok = true;
    for (int64_t u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
      const Fp4Unit U = fp4_unit(p, u);
      if (U.tile_begin >= U.tile_end) continue;
      if (!(ok = esync())) break;  // everyone is done with the previous unit's tables
      if (do_hist && U.row != hist_row) {
        if (hist_row >= 0) flush_hist(true);
        hist_row = U.row;
      }
      // the unit's query block scales (as floats) and head weights
      {
        const uint8_t* qsb = p.qI_scale + U.row * (kHeads * 4);
        for (int i = et; i < kHeads * 4; i += kEpiThreads) qs_t[i] = e8m0_value(__ldg(qsb + i));
        for (int i = et; i < kHeads; i += kEpiThreads) {
          uint32_t mx, mn;
          exp_range(__ldg(reinterpret_cast<const uint32_t*>(qsb) + i), mx, mn);
          w_t[i] = __ldg(p.w + U.row * kHeads + i);
          wq_t[i] = w_t[i] * e8m0_value(mx);
        }
      }
      if (!(ok = esync())) break;
      const int64_t vis = visible_checked(query_pos(p.q_pos, p.q_pos0, U.row, U.j), p.m, p.n_entries, p.dev_status,
                                          lane == 0 && U.tile_begin == 0);
      for (int64_t t = U.tile_begin; t < U.tile_end; ++t, ++seq) {
        if ((int)(seq % kEpiGroups) != grp) continue;  // another group's tile
        const int a = (int)(seq % kAcc), r = (int)(seq % kScaleRing);
        if (!(ok = tc::mbar_wait(&bars[kBarKsFull + r], (uint32_t)((seq / kScaleRing) & 1), s_abort, 13))) break;
        const int row = quad * 32 + lane;
        const int64_t s = t * kTileE + row;
        const uint32_t kw = ks_ring[r * kTileE + row];
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * kHeads);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        // one turn of the slot: wait for its product; once it is read, release the slot
        auto turn_wait = [&]() -> bool {
          if (!tc::mbar_wait(&bars[kBarAccFull + a], (tpar >> a) & 1u, s_abort, 12)) return false;
          tc::tc_fence_after();
          return true;
        };
        auto turn_release = [&]() {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bars[kBarAccEmpty + a]);
          tpar ^= 1u << a;
        };
        if (tile_fast[r]) {
          // folded tile: S[e,h] * 2^(Rk[e] - 127) * 2^(Rq[h] - 127); the two powers of two
          // are positive and exact, so 2^(Rk[e] - 127) * sum_h (w[h] 2^(Rq[h] - 127)) ReLU(S[e,h])
          if (!(ok = turn_wait())) break;
          float v0[32], v1[32];
          tc::tmem_ld32(taddr, v0);
          tc::tmem_ld32(taddr + 32u, v1);
          tc::tmem_ld_wait();
          turn_release();
          const float4* wq4 = reinterpret_cast<const float4*>(wq_t);
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 c = wq4[h4];
            ps[0] = fmaf(c.x, fmaxf(v0[4 * h4 + 0], 0.f), ps[0]);
            ps[1] = fmaf(c.y, fmaxf(v0[4 * h4 + 1], 0.f), ps[1]);
            ps[2] = fmaf(c.z, fmaxf(v0[4 * h4 + 2], 0.f), ps[2]);
            ps[3] = fmaf(c.w, fmaxf(v0[4 * h4 + 3], 0.f), ps[3]);
          }
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 c = wq4[8 + h4];
            ps[0] = fmaf(c.x, fmaxf(v1[4 * h4 + 0], 0.f), ps[0]);
            ps[1] = fmaf(c.y, fmaxf(v1[4 * h4 + 1], 0.f), ps[1]);
            ps[2] = fmaf(c.z, fmaxf(v1[4 * h4 + 2], 0.f), ps[2]);
            ps[3] = fmaf(c.w, fmaxf(v1[4 * h4 + 3], 0.f), ps[3]);
          }
          uint32_t mx, mn;
          exp_range(kw, mx, mn);
          const float kr = e8m0_value(mx);
#pragma unroll
          for (int i = 0; i < 4; ++i) ps[i] *= kr;
        } else {
          // blocked tile: the four blocks' products (one turn each), each with its two scales
          float dot[kHeads];
#pragma unroll
          for (int h = 0; h < kHeads; ++h) dot[h] = 0.f;
          for (int k = 0; k < 4 && ok; ++k) {
            if (!(ok = turn_wait())) break;
            const float ksk = e8m0_value((kw >> (8 * k)) & 0xFFu);
#pragma unroll
            for (int hb = 0; hb < kHeads; hb += 32) {
              float v[32];
              tc::tmem_ld32(taddr + (uint32_t)hb, v);
              tc::tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < 32; ++h) dot[hb + h] = fmaf(v[h] * ksk, qs_t[(hb + h) * 4 + k], dot[hb + h]);
            }
            turn_release();
          }
          if (!ok) break;
#pragma unroll
          for (int h = 0; h < kHeads; ++h) ps[h & 3] = fmaf(w_t[h], fmaxf(dot[h], 0.f), ps[h & 3]);
        }
        const float score = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars[kBarKsEmpty + r]);
        const bool keep = s < vis;
        if (keep) p.scores[U.row * p.score_stride + s] = score;
        if (do_hist) {
          // lanes with the same bin add their count once (scores crowd into few bins)
          const uint32_t bin = keep ? float_order_key(score) >> (32 - kTopkHistBits) : 0xFFFFFFFFu;
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (keep && lane == __ffs(peers) - 1) atomicAdd(&hist[bin >> 1], (uint32_t)__popc(peers) << (16 * (bin & 1)));
        }
      }
    }
    if (do_hist && ok && hist_row >= 0 && esync()) flush_hist(false);
  }

  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) flag_status(p.dev_status, HYB_DEV_TIMEOUT | ((*s_abort & 0xFF) << 8));
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool index_fp4_shape_supported(const hyb_index_args* a) {
  if (a->dtype != HYB_MXFP4 || a->c_I != 128 || a->n_ih != kHeads) return false;
  const int64_t kvs = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  if (kvs % 4 != 0) return false;  // rows of scale words start on 16-byte boundaries
  const uintptr_t al = reinterpret_cast<uintptr_t>(a->kI) | reinterpret_cast<uintptr_t>(a->kI_scale) |
                       reinterpret_cast<uintptr_t>(a->qI) | reinterpret_cast<uintptr_t>(a->qI_scale);
  if (al % 16 != 0) return false;
  if (a->batch * kvs >= (int64_t(1) << 31) || a->batch * a->n_q * kHeads >= (int64_t(1) << 31)) return false;
  return true;
}

cudaError_t launch_index_scores_fp4(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                    uint32_t* ghist, bool* hist_done, cudaStream_t s) {
  *hist_done = false;
  if (n_vis_max == 0 || a->n_q == 0 || a->batch == 0) return cudaSuccess;
  const int64_t kvs = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  CUtensorMap tm_keys, tm_ks, tm_q;
  if (!encode_tmap_2d(&tm_keys, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->kI, kRowRaw, (uint64_t)(a->batch * kvs), kRowRaw,
                      kRowRaw, kTileE, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&tm_ks, CU_TENSOR_MAP_DATA_TYPE_UINT32, a->kI_scale, (uint64_t)kvs, (uint64_t)a->batch,
                      (uint64_t)kvs * 4, kTileE, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->qI, kRowRaw, (uint64_t)(a->batch * a->n_q * kHeads),
                      kRowRaw, kRowRaw, kHeads, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  Fp4Params p{};
  p.w = a->w, p.qI_scale = reinterpret_cast<const uint8_t*>(a->qI_scale), p.scores = scores;
  p.score_stride = score_stride;
  p.n_q = a->n_q, p.n_entries = a->n_entries, p.kv_stride = kvs, p.m = a->m, p.q_pos0 = a->q_pos0;
  p.q_pos = a->q_pos;
  p.dev_status = a->dev_status;
  const int64_t rows = a->batch * a->n_q;
  const int64_t tiles_max = (n_vis_max + kTileE - 1) / kTileE;
  // one unit per CTA where the rows are few (decode), the runs evened out over the SMs
  int64_t tpu = (rows * tiles_max + kNumSMs - 1) / kNumSMs;
  tpu = tpu < 1 ? 1 : (tpu > tiles_max ? tiles_max : tpu);
  p.tiles_per_unit = tpu;
  p.units_per_group = (tiles_max + tpu - 1) / tpu;
  p.n_units = rows * p.units_per_group;
  // fused histogram: fewer than 2^16 entries per unit (16-bit counters)
  p.ghist = (ghist != nullptr && tpu * kTileE < 65536) ? ghist : nullptr;
  cudaError_t e = cudaFuncSetAttribute(index_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.n_units < kNumSMs ? p.n_units : kNumSMs;
  e = launch_pdl(index_fp4_kernel, dim3((unsigned)grid), dim3(kThreads), (size_t)kSmemBytes, s, tm_keys, tm_ks, tm_q, p);
  if (e != cudaSuccess) return e;
  *hist_done = p.ghist != nullptr;
  return cudaGetLastError();
}

}  // namespace hyb
