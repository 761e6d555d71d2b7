// topk.cu -- top-k selector of the lightning indexer ("DeepSeek-V4 hybrid
// attention" (trishampatil.com) section V.2: the k best-scoring compressed
// blocks are kept; "DeepSeek-V4: Anatomy..." (modernaiengineering.com) worked
// example: fewer than k entries are kept when fewer exist).
//
// Ranking: (score descending, entry index ascending), compared exactly on the
// order-preserving uint32 image ("key") of the float32 scores.  The kept set
// is every entry with key > T plus the lowest-indexed entries with key == T,
// where T is the k-th largest key; it is written in ascending index order and
// padded with -1.
//
// Building blocks (CTAs of 1024 threads):
//   radix_select     exact k-th key of a list, 8 bits per pass from the top;
//                    histogram atomics are aggregated per warp (match.any), so
//                    lists whose keys share their top bits do not serialise.
//   collect_ordered  one pass in list order that writes the kept positions to
//                    their final (ascending) slots: a block scan of the
//                    (key > T, key == T) flags gives each kept element's slot,
//                    so no sort is needed.
// Plans:
//   one stage   (rows of at most kStageCap visible entries, unless few rows of more
//               than kGridMinEntries take the grid plan): one CTA per row stages the
//               keys in shared memory, selects and collects.
//   three kernels (longer rows, e.g. 262,144 entries at 1M context):
//     hist    CTA (chunk, row): 12-bit histogram of its chunk, added into the
//             row's global histogram (the tensor-core indexer builds it in its
//             epilogue for decode rows; then this kernel is skipped).
//     filter  CTA (chunk, row): from the row histogram, the bin b* that holds
//             the k-th largest key; the chunk's entries above b* (all kept)
//             and inside b* (candidates) are written, in index order, to the
//             chunk's own regions.
//             The filter also histograms the next 12 bits of the candidates.
//     final   (the row's last filter CTA): from that second histogram, the digit b2 holding
//             the last kept candidate; candidates above it are kept, the few
//             equal to it are selected exactly; the kept candidates are then
//             merged with the entries above b* (both lists are ascending).
//   grid (decode: at most one row per SM, up to kGridChunkCap entries per CTA):
//             one kernel whose CTAs are all resident at once (at most one CTA
//             per SM, and one fits).  CTA (part, row) stages its chunk of the
//             row's keys in shared memory once; the CTAs agree on the threshold
//             through global histograms, with a grid-wide barrier between phases:
//       1  b1 = the 12-bit bin holding the k-th largest key (row histogram);
//          the chunk's keys in b1 are histogrammed on their next 12 bits.
//       2  b2 = the second-level bin holding the last kept key.  Keys whose top
//          24 bits are above (b1, b2) are kept; the few whose top 24 bits equal
//          it (sub-candidates) go to the row's list; every CTA publishes how
//          many of its keys are surely kept.
//       3  every CTA ranks the row's list by (key desc, entry asc) and keeps the
//          r2 best, then writes its kept entries in ascending order at the
//          offset given by the counts of the CTAs before it.
//          When a row's list overflows (many keys share their top 24 bits), all
//          CTAs take two more barriers: a histogram of the last 8 bits gives the
//          exact k-th key T, and the keys equal to T are kept lowest entry first
//          through a prefix of the tie counts over the CTAs.
#include "kernels.cuh"

namespace hyb {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int64_t kStageCap = 16384;  // one-stage plan: keys staged in shared memory
constexpr int64_t kCandCap = 65536;   // final kernel: candidates tracked by a shared-memory bitmap
constexpr int64_t kSubCap = 8192;     // final kernel: second-level candidates staged in shared memory
constexpr int kRun = 8;               // final kernel: candidates per thread per round
constexpr int kHistBits = kTopkHistBits;
constexpr int kHistBins = kTopkHistBins;
constexpr int kMaxChunks = 64;
constexpr int kPer = 8;  // keys a thread loads before using them (histogram and filter passes)
constexpr int64_t kGridChunkCap = 32768;  // grid plan: keys per CTA, staged in shared memory
constexpr int64_t kGridMinEntries = 4096; // shorter rows always take the one-stage plan
constexpr int kCandListCap = 4096;        // grid plan: candidates per row selected in shared memory
constexpr int kSubListCap = 1024;         // grid plan, overflow: sub-candidates per row ranked directly
constexpr int kGridSlot = 8;              // grid plan: published counts per CTA

struct TopkParams {
  const float* scores;
  int64_t score_stride;
  int32_t* idx;
  float* out_scores;
  int64_t n_q, n_entries, m, k, q_pos0;
  const int64_t* q_pos;  // optional per-query positions [rows]
  // three-kernel plan
  int64_t chunk;
  int n_chunks;
  uint32_t* ghist;      // [rows][kHistBins]: first digit (top kHistBits of the key) of every score
  uint32_t* ghist2;     // [rows][kHistBins]: second digit of the threshold bin's candidates
  int32_t* def_idx;     // [rows][n_chunks][chunk]: entries above the threshold bin
  uint32_t* cand_key;   // [rows][n_chunks][chunk]: entries in the threshold bin
  int32_t* cand_idx;
  int32_t* counts;      // [rows][n_chunks][2]: (#above, #candidates) of each chunk
  uint32_t* done;       // [rows]: filter CTAs finished (the last one selects)
  // grid plan (ghist, ghist2 and chunk/n_chunks as above)
  uint32_t* hist3;      // [rows][256]: last 8 bits of the sub-candidates (overflow only)
  uint32_t* nsub;       // [rows]: sub-candidates appended to the row's sub-list
  uint32_t* ncand;      // [rows]: candidates appended to the row's list
  uint32_t* dep;        // [rows]: CTAs of the row that finished
  uint32_t* gsync;      // [0]: grid-barrier arrivals, [1]: a sub-list overflowed, [2]: CTAs that finished
  int32_t* slots;       // [rows][n_chunks][kGridSlot]: published per-CTA counts (slow path 0-2, list 4-6)
  uint2* cand;          // [rows][n_chunks][chunk]: (key, entry) of each CTA's first-level candidates
  uint2* sub;           // [rows][kSubListCap]: (key, entry) of the sub-candidates
  int hist_done;        // the row histograms were filled by the indexer
  int32_t* dev_status;
  long long wait_cycles;  // bound of a grid-barrier wait (SM clock cycles)
};

// (a bad device-side position was reported by the scoring kernel of the same call)
__device__ __forceinline__ int64_t row_visible(const TopkParams& p, int64_t row) {
  const int64_t j = row % p.n_q;
  return visible_checked(query_pos(p.q_pos, p.q_pos0, row, j), p.m, p.n_entries, nullptr, false);
}

struct BlockShared {
  uint32_t hist[256];
  uint32_t warp_tot[kTopkWarps];
  uint32_t total;
  uint32_t prefix, mask, desired;
};

// Exclusive block-wide prefix of two flags packed as (a | b << 16) in thread
// order; returns (a_before, b_before) of this thread and the block totals.
__device__ __forceinline__ void block_scan2(bool fa, bool fb, BlockShared& S, uint32_t& a_before, uint32_t& b_before,
                                            uint32_t& a_tot, uint32_t& b_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ba = __ballot_sync(0xffffffffu, fa), bb = __ballot_sync(0xffffffffu, fb);
  const uint32_t lt = (1u << lane) - 1u;
  if (lane == 0) S.warp_tot[warp] = (uint32_t)__popc(ba) | ((uint32_t)__popc(bb) << 16);
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = S.warp_tot[lane];
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    S.warp_tot[lane] = incl - v;
    if (lane == 31) S.total = incl;
  }
  __syncthreads();
  const uint32_t base = S.warp_tot[warp];
  a_before = (base & 0xFFFFu) + (uint32_t)__popc(ba & lt);
  b_before = (base >> 16) + (uint32_t)__popc(bb & lt);
  a_tot = S.total & 0xFFFFu;
  b_tot = S.total >> 16;
  __syncthreads();
}

// Exclusive block-wide prefix of two per-thread counts (each block total < 2^16)
// in thread order; returns this thread's (a_before, b_before) and the totals.
__device__ __forceinline__ void block_scan_counts(uint32_t a, uint32_t b, BlockShared& S, uint32_t& a_before,
                                                  uint32_t& b_before, uint32_t& a_tot, uint32_t& b_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t v = a | (b << 16);
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) S.warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = S.warp_tot[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    S.warp_tot[lane] = wi - w;
    if (lane == 31) S.total = wi;
  }
  __syncthreads();
  const uint32_t base = S.warp_tot[warp] + incl - v;
  a_before = base & 0xFFFFu;
  b_before = base >> 16;
  a_tot = S.total & 0xFFFFu;
  b_tot = S.total >> 16;
  __syncthreads();
}

__device__ __forceinline__ void hist_add(uint32_t* hist, bool take, uint32_t digit) {
  const uint32_t active = __ballot_sync(0xffffffffu, take);
  if (take) {
    const uint32_t peers = __match_any_sync(active, digit);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
  }
}

// The `take`-th largest key T of keyfn(0..L) and how many elements equal to T
// are kept (the lowest positions).  Requires 1 <= take <= L.
template <typename KeyFn>
__device__ void radix_select(KeyFn keyfn, int64_t L, int64_t take, BlockShared& S, uint32_t& T, uint32_t& ties) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) S.prefix = 0, S.mask = 0, S.desired = (uint32_t)take;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) S.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = S.prefix, mask = S.mask;
    for (int64_t base = 0; base < L; base += kTopkThreads) {
      const int64_t s = base + tid;
      const uint32_t key = s < L ? keyfn(s) : 0u;
      hist_add(S.hist, s < L && (key & mask) == prefix, (key >> shift) & 255u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l covers digits hi..hi-7 with hi = 255 - 8l (lane 0 = largest digits)
      const int hi = 255 - 8 * lane;
      uint32_t lane_sum = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) lane_sum += S.hist[hi - d];
      uint32_t incl = lane_sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - lane_sum;
      const uint32_t desired = S.desired;
      if (excl < desired && desired <= incl) {
        uint32_t cum = excl;
        for (int d = hi; d > hi - 8; --d) {
          if (cum + S.hist[d] >= desired) {
            S.prefix = prefix | ((uint32_t)d << shift);
            S.mask = mask | (255u << shift);
            S.desired = desired - cum;
            break;
          }
          cum += S.hist[d];
        }
      }
    }
    __syncthreads();
  }
  T = S.prefix;
  ties = S.desired;
  __syncthreads();
}

// Calls emit(slot, position) for every kept position, slot = its rank in list
// order among the kept ones (0 .. take-1).
template <typename KeyFn, typename Emit>
__device__ void collect_ordered(KeyFn keyfn, int64_t L, uint32_t T, uint32_t ties, BlockShared& S, Emit emit) {
  uint32_t gt_base = 0, eq_base = 0;
  for (int64_t base = 0; base < L; base += kTopkThreads) {
    const int64_t s = base + threadIdx.x;
    const uint32_t key = s < L ? keyfn(s) : 0u;
    const bool gt = s < L && key > T;
    const bool eq = s < L && key == T;
    uint32_t gb, eb, gtot, etot;
    block_scan2(gt, eq, S, gb, eb, gtot, etot);
    gb += gt_base, eb += eq_base;
    if (gt) emit(gb + (eb < ties ? eb : ties), s);
    if (eq && eb < ties) emit(gb + eb, s);
    gt_base += gtot, eq_base += etot;
  }
}

__device__ __forceinline__ void keep_all(const TopkParams& p, int64_t row, int64_t vis) {
  const float* sc = p.scores + row * p.score_stride;
  int32_t* out = p.idx + row * p.k;
  float* out_sc = p.out_scores ? p.out_scores + row * p.k : nullptr;
  for (int64_t i = threadIdx.x; i < p.k; i += kTopkThreads) {
    out[i] = i < vis ? (int32_t)i : -1;
    if (out_sc) out_sc[i] = i < vis ? sc[i] : -INFINITY;
  }
}

// ------------------------------------------------------------- one stage
__global__ void __launch_bounds__(kTopkThreads) topk_row_kernel(TopkParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t keys_s[];  // [kStageCap]
  __shared__ BlockShared S;
  const int64_t row = blockIdx.x;
  const int64_t vis = row_visible(p, row);
  if (vis <= p.k) {
    keep_all(p, row, vis);
    return;
  }
  const float* sc = p.scores + row * p.score_stride;
  int32_t* out = p.idx + row * p.k;
  float* out_sc = p.out_scores ? p.out_scores + row * p.k : nullptr;
  for (int64_t s = threadIdx.x; s < vis; s += kTopkThreads) keys_s[s] = float_order_key(__ldg(sc + s));
  __syncthreads();
  auto keyfn = [&](int64_t s) { return keys_s[s]; };
  uint32_t T, ties;
  radix_select(keyfn, vis, p.k, S, T, ties);
  collect_ordered(keyfn, vis, T, ties, S, [&](uint32_t slot, int64_t s) {
    out[slot] = (int32_t)s;
    if (out_sc) out_sc[slot] = sc[s];
  });
}

// ------------------------------------------------ three kernels: hist
__global__ void __launch_bounds__(kTopkThreads) topk_hist_kernel(TopkParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t hist[kHistBins];
  const int64_t row = blockIdx.y;
  const int64_t vis = row_visible(p, row);
  if (vis <= p.k) return;
  const int64_t s0 = (int64_t)blockIdx.x * p.chunk;
  if (s0 >= vis) return;
  const int64_t len = vis - s0 < p.chunk ? vis - s0 : p.chunk;
  for (int i = threadIdx.x; i < kHistBins; i += kTopkThreads) hist[i] = 0;
  __syncthreads();
  const float* sc = p.scores + row * p.score_stride + s0;
  for (int64_t base = 0; base < len; base += kPer * kTopkThreads) {
    uint32_t key[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {  // all loads first: one round trip per kPer elements
      const int64_t s = base + u * kTopkThreads + threadIdx.x;
      key[u] = s < len ? float_order_key(__ldg(sc + s)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      hist_add(hist, base + u * kTopkThreads + threadIdx.x < len, key[u] >> (32 - kHistBits));
  }  __syncthreads();
  uint32_t* gh = p.ghist + row * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kTopkThreads)
    if (hist[i]) atomicAdd(gh + i, hist[i]);
}

// The bin holding the k-th largest key of a row, from its histogram, and the
// number of keys in higher bins (< k).
__device__ void threshold_bin(const uint32_t* gh, uint32_t k, BlockShared& S, uint32_t& bstar, uint32_t& above) {
  constexpr int kPer = kHistBins / kTopkThreads;  // bins per thread, from the top
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hi = kHistBins - 1 - kPer * tid;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int d = 0; d < kPer; ++d) c[d] = gh[hi - d], sum += c[d];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) S.warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = S.warp_tot[lane];
    uint32_t wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    S.warp_tot[lane] = wi - v;
  }
  __syncthreads();
  const uint32_t excl = S.warp_tot[warp] + incl - sum;  // keys in bins above this thread's
  if (excl < k && k <= excl + sum) {
    uint32_t cum = excl;
    for (int d = 0; d < kPer; ++d) {
      if (cum + c[d] >= k) {
        S.prefix = (uint32_t)(hi - d);
        S.desired = cum;
        break;
      }
      cum += c[d];
    }
  }
  __syncthreads();
  bstar = S.prefix;
  above = S.desired;
  __syncthreads();
}

// ------------------------------------------ three kernels: final selection
// Run by the last filter CTA of a row, once every chunk's lists and counts are final.
__device__ void final_select(const TopkParams& p, int64_t row, uint32_t* dyn, BlockShared& S) {
  __shared__ int32_t pre_d[kMaxChunks + 1], pre_c[kMaxChunks + 1];
  const int64_t vis = row_visible(p, row);
  if (vis <= p.k) {
    keep_all(p, row, vis);
    return;
  }
  const int tid = threadIdx.x;
  const float* sc = p.scores + row * p.score_stride;
  int32_t* out = p.idx + row * p.k;
  float* out_sc = p.out_scores ? p.out_scores + row * p.k : nullptr;
  const int32_t* cnt = p.counts + row * p.n_chunks * 2;
  // prefix sums of the per-chunk counts (at most 64 chunks: two per lane of warp 0)
  if (tid < 32) {
    int32_t d[2], c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = h * 32 + tid;
      d[h] = ch < p.n_chunks ? cnt[2 * ch] : 0;
      c[h] = ch < p.n_chunks ? cnt[2 * ch + 1] : 0;
    }
    int32_t carry_d = 0, carry_c = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int32_t id = d[h], ic = c[h];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t ud = __shfl_up_sync(0xffffffffu, id, o), uc = __shfl_up_sync(0xffffffffu, ic, o);
        if (tid >= o) id += ud, ic += uc;
      }
      pre_d[h * 32 + tid + 1] = carry_d + id;
      pre_c[h * 32 + tid + 1] = carry_c + ic;
      carry_d += __shfl_sync(0xffffffffu, id, 31);
      carry_c += __shfl_sync(0xffffffffu, ic, 31);
    }
    if (tid == 0) pre_d[0] = 0, pre_c[0] = 0;
  }
  __syncthreads();
  const int64_t n_def = pre_d[p.n_chunks], n_cand = pre_c[p.n_chunks];
  const int64_t r = p.k - n_def;  // candidates to keep (>= 1)
  const int64_t reg0 = row * p.n_chunks * p.chunk;
  int32_t* A = reinterpret_cast<int32_t*>(dyn);  // [k]: entries above the threshold bin, ascending
  int32_t* B = A + p.k;                          // [k]: kept candidates, ascending
  uint32_t* sk = reinterpret_cast<uint32_t*>(B + p.k);  // [kSubCap] keys of the sub-candidates
  int32_t* spos = reinterpret_cast<int32_t*>(sk + kSubCap);  // [kSubCap] their candidate positions
  uint32_t* selbits = reinterpret_cast<uint32_t*>(spos + kSubCap);  // [kCandCap/32] selected sub-candidates
  // chunk holding element x of a concatenated list: the last c with pre[c] <= x
  auto chunk_in = [&](const int32_t* pre, int64_t x) {
    int lo = 0, hi = p.n_chunks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  auto cand_at = [&](int64_t x) { const int c = chunk_in(pre_c, x); return reg0 + (int64_t)c * p.chunk + (x - pre_c[c]); };
  for (int64_t x = tid; x < n_def; x += kTopkThreads) {
    const int c = chunk_in(pre_d, x);
    A[x] = p.def_idx[reg0 + (int64_t)c * p.chunk + (x - pre_d[c])];
  }
  // second-level threshold among the candidates: digit2 = the next kHistBits of the key
  uint32_t b2, above2;
  threshold_bin(p.ghist2 + row * kHistBins, (uint32_t)r, S, b2, above2);
  const int64_t r2 = r - above2;  // how many of the candidates with digit2 == b2 to keep
  auto digit2 = [&](uint32_t key) { return (key >> (32 - 2 * kHistBits)) & (uint32_t)(kHistBins - 1); };
  // Passes over the candidates in rounds of kRun * kTopkThreads: in a round each thread
  // takes a contiguous run of kRun candidates and loads them all at once (one round trip
  // per round), and one block scan orders the round.
  const bool fast = n_cand <= kCandCap;
  constexpr int64_t kRound = (int64_t)kRun * kTopkThreads;
  // global offsets of a run's candidates: chunks first (shared memory only), so that
  // the loads that follow are all independent
  auto run_offsets = [&](int64_t x0, int64_t x1, int64_t (&at)[kRun]) {
    int c = x0 < n_cand ? chunk_in(pre_c, x0) : 0;
#pragma unroll
    for (int u = 0; u < kRun; ++u) {
      const int64_t x = x0 + u;
      if (x < x1) {
        while (pre_c[c + 1] <= x) ++c;  // a run crosses chunk boundaries in order
        at[u] = reg0 + (int64_t)c * p.chunk + (x - pre_c[c]);
      } else {
        at[u] = 0;
      }
    }
  };
  auto load_run = [&](int64_t base, uint32_t (&rk)[kRun], int64_t& x0, int64_t& x1) {
    x0 = std::min<int64_t>(base + (int64_t)tid * kRun, n_cand);
    x1 = std::min<int64_t>(x0 + kRun, n_cand);
    int64_t at[kRun];
    run_offsets(x0, x1, at);
#pragma unroll
    for (int u = 0; u < kRun; ++u) rk[u] = x0 + u < x1 ? p.cand_key[at[u]] : 0u;
  };
  uint32_t n_sub = 0;
  if (fast) {
    // the sub-candidates (digit2 == b2), in candidate order
    for (int64_t base = 0; base < n_cand; base += kRound) {
      uint32_t rk[kRun];
      int64_t x0, x1;
      load_run(base, rk, x0, x1);
      uint32_t mine = 0;
#pragma unroll
      for (int u = 0; u < kRun; ++u) mine += (x0 + u < x1 && digit2(rk[u]) == b2);
      uint32_t sb, zb, st, zt;
      block_scan_counts(mine, 0u, S, sb, zb, st, zt);
      sb += n_sub;
#pragma unroll
      for (int u = 0; u < kRun; ++u)
        if (x0 + u < x1 && digit2(rk[u]) == b2) {
          if (sb < kSubCap) sk[sb] = rk[u], spos[sb] = (int32_t)(x0 + u);
          ++sb;
        }
      n_sub += st;
    }
  }
  if (fast && n_sub <= kSubCap) {
    for (int64_t x = tid; x < kCandCap / 32; x += kTopkThreads) selbits[x] = 0u;
    __syncthreads();
    auto mark = [&](int64_t x) {
      const int32_t pos = spos[x];
      atomicOr(&selbits[pos >> 5], 1u << (pos & 31));
    };
    if (r2 == n_sub) {  // every sub-candidate is kept
      for (int64_t x = tid; x < n_sub; x += kTopkThreads) mark(x);
    } else if (n_sub <= kTopkThreads) {
      // few: rank each directly by (key desc, position asc); the r2 best are kept
      if (tid < n_sub) {
        const uint32_t kx = sk[tid];
        int64_t rank = 0;
        for (int64_t y = 0; y < n_sub; ++y) {
          const uint32_t ky = sk[y];
          rank += ky > kx || (ky == kx && y < tid);
        }
        if (rank < r2) mark(tid);
      }
    } else {
      uint32_t T, ties;
      auto subkey = [&](int64_t x) { return sk[x]; };
      radix_select(subkey, n_sub, r2, S, T, ties);
      collect_ordered(subkey, n_sub, T, ties, S, [&](uint32_t, int64_t x) { mark(x); });
    }
    __syncthreads();
    // kept candidates in order: digit2 above b2, or selected among the sub-candidates
    uint32_t nb = 0;
    for (int64_t base = 0; base < n_cand; base += kRound) {
      uint32_t rk[kRun];
      int64_t x0, x1;
      load_run(base, rk, x0, x1);
      bool keep[kRun];
      uint32_t mine = 0;
#pragma unroll
      for (int u = 0; u < kRun; ++u) {
        const int64_t x = x0 + u;
        const uint32_t d2 = x < x1 ? digit2(rk[u]) : 0u;
        keep[u] = x < x1 && (d2 > b2 || (d2 == b2 && ((selbits[x >> 5] >> (x & 31)) & 1u)));
        mine += keep[u];
      }
      uint32_t kb, zb, kt, zt;
      block_scan_counts(mine, 0u, S, kb, zb, kt, zt);
      kb += nb;
      int64_t at[kRun];
      run_offsets(x0, x1, at);
      int32_t ix[kRun];
#pragma unroll
      for (int u = 0; u < kRun; ++u) ix[u] = keep[u] ? p.cand_idx[at[u]] : 0;
#pragma unroll
      for (int u = 0; u < kRun; ++u)
        if (keep[u]) B[kb++] = ix[u];
      nb += kt;
    }
  } else {
    // many equal keys: exact selection over all candidates, read in place
    auto inplace = [&](int64_t x) { return p.cand_key[cand_at(x)]; };
    uint32_t T, ties;
    radix_select(inplace, n_cand, r, S, T, ties);
    collect_ordered(inplace, n_cand, T, ties, S, [&](uint32_t slot, int64_t x) { B[slot] = p.cand_idx[cand_at(x)]; });
  }
  __syncthreads();
  // merge the two ascending, disjoint lists: slot = own rank + rank in the other list
  for (int64_t x = tid; x < n_def + r; x += kTopkThreads) {
    const bool in_a = x < n_def;
    const int32_t v = in_a ? A[x] : B[x - n_def];
    const int32_t* other = in_a ? B : A;
    int64_t lo = 0, hi = in_a ? r : n_def;  // count of elements of `other` below v
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (other[mid] < v) lo = mid + 1; else hi = mid;
    }
    const int64_t slot = (in_a ? x : x - n_def) + lo;
    out[slot] = v;
    if (out_sc) out_sc[slot] = sc[v];
  }
}

// ---------------------------------------------- three kernels: filter
__device__ void filter_chunk(const TopkParams& p, int64_t row, int64_t vis, BlockShared& S);

// Every CTA filters its chunk, then counts itself done; the row's last CTA (no
// waiting: it is simply the one that finds all others done) runs the final selection.
__global__ void __launch_bounds__(kTopkThreads) topk_filter_kernel(TopkParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t dyn[];
  __shared__ BlockShared S;
  __shared__ uint32_t s_last;
  const int64_t row = blockIdx.y;
  const int64_t vis = row_visible(p, row);
  if (vis > p.k) filter_chunk(p, row, vis, S);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(p.done + row, 1u) == (uint32_t)(p.n_chunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  final_select(p, row, dyn, S);
}

__device__ void filter_chunk(const TopkParams& p, int64_t row, int64_t vis, BlockShared& S) {
  const int64_t s0 = (int64_t)blockIdx.x * p.chunk;
  int32_t* cnt = p.counts + (row * p.n_chunks + blockIdx.x) * 2;
  if (s0 >= vis) {
    if (threadIdx.x == 0) cnt[0] = 0, cnt[1] = 0;
    return;
  }
  const int64_t len = vis - s0 < p.chunk ? vis - s0 : p.chunk;
  __shared__ uint32_t hist2[kHistBins];  // 16 KiB
  for (int i = threadIdx.x; i < kHistBins; i += kTopkThreads) hist2[i] = 0;
  uint32_t bstar, above;
  threshold_bin(p.ghist + row * kHistBins, (uint32_t)p.k, S, bstar, above);  // (syncs the zeroing too)
  const float* sc = p.scores + row * p.score_stride + s0;
  const int64_t reg = (row * p.n_chunks + blockIdx.x) * p.chunk;
  // each thread takes 4 consecutive entries, so one block scan orders 4096 of them
  uint32_t nd = 0, nc = 0;
  for (int64_t base = 0; base < len; base += 4 * kTopkThreads) {
    const int64_t s = base + 4 * threadIdx.x;
    uint32_t key[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) key[u] = s + u < len ? float_order_key(__ldg(sc + s + u)) : 0u;
    bool d[4], c[4];
    uint32_t ld = 0, lc = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t bin = key[u] >> (32 - kHistBits);
      d[u] = s + u < len && bin > bstar;
      c[u] = s + u < len && bin == bstar;
      ld += d[u], lc += c[u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) hist_add(hist2, c[u], (key[u] >> (32 - 2 * kHistBits)) & (kHistBins - 1));
    uint32_t db, cb, dt, ct;
    block_scan_counts(ld, lc, S, db, cb, dt, ct);
    uint32_t od = nd + db, oc = nc + cb;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (d[u]) p.def_idx[reg + od++] = (int32_t)(s0 + s + u);
      if (c[u]) {
        p.cand_key[reg + oc] = key[u];
        p.cand_idx[reg + oc++] = (int32_t)(s0 + s + u);
      }
    }
    nd += dt, nc += ct;
  }
  if (threadIdx.x == 0) cnt[0] = (int32_t)nd, cnt[1] = (int32_t)nc;
  __syncthreads();
  uint32_t* gh2 = p.ghist2 + row * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kTopkThreads)
    if (hist2[i]) atomicAdd(gh2 + i, hist2[i]);
}


// ------------------------------------------------------------------ grid plan
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// Barrier over all CTAs of the grid.  Arrivals count up in *count (zeroed before
// the launch), so the i-th barrier waits for i * gridDim.x * gridDim.y of them.
// Bounded: on expiry HYB_DEV_TIMEOUT (with the site) is raised and false returned.
__device__ bool grid_barrier(uint32_t* count, uint32_t target, int32_t* dev_status, int site, long long limit) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(count, 1u);
    int ok = 1;
    const long long t0 = clock64();
    while (ld_acquire_u32(count) < target) {
      if (clock64() - t0 > limit) {
        ok = 0;
        break;
      }
    }
    if (!ok) flag_status(dev_status, HYB_DEV_TIMEOUT | (site << 8));
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// The float32 whose order-preserving key is k (the inverse of float_order_key; -0 comes back as +0).
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Sum over the CTA of one value per thread (every thread gets the total).
__device__ __forceinline__ uint32_t block_sum(uint32_t v, BlockShared& S) {
  uint32_t before, z0, tot, z1;
  block_scan_counts(v, 0u, S, before, z0, tot, z1);
  return tot;
}

__global__ void __launch_bounds__(kTopkThreads, 1) topk_grid_kernel(TopkParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t dyn[];
  uint32_t* keys = dyn;                                           // [chunk] keys of this CTA's entries
  uint32_t* hist = keys + p.chunk;                                // [kHistBins]
  uint2* list = reinterpret_cast<uint2*>(hist + kHistBins);       // [kSubListCap] the row's sub-candidates
  uint32_t* selb = reinterpret_cast<uint32_t*>(list + kSubListCap);  // [chunk / 32] selected sub-candidates
  uint2* sorted = reinterpret_cast<uint2*>(selb + p.chunk / 32);     // [kCandListCap] candidates by entry
  uint32_t* kbits = reinterpret_cast<uint32_t*>(sorted + kCandListCap);  // [kCandListCap / 32] kept ones
  __shared__ BlockShared S;
  __shared__ int64_t s_before;
  const int tid = threadIdx.x;
  const int part = blockIdx.x, parts = gridDim.x;
  const int64_t row = blockIdx.y;
  const uint32_t nblk = gridDim.x * gridDim.y;
  uint32_t nbar = 0;
  const int64_t vis = row_visible(p, row);
  const int64_t s0 = (int64_t)part * p.chunk;
  const int64_t len = vis - s0 < 0 ? 0 : (vis - s0 < p.chunk ? vis - s0 : p.chunk);
  const bool active = vis > p.k;  // rows with at most k visible entries keep them all
  const float* sc = p.scores + row * p.score_stride;
  int32_t* out = p.idx + row * p.k;
  float* out_sc = p.out_scores ? p.out_scores + row * p.k : nullptr;
  int32_t* myslot = p.slots + ((int64_t)row * parts + part) * kGridSlot;
  // each thread owns a contiguous run of the chunk, so block scans keep entry order
  const int per = (int)(p.chunk / kTopkThreads);
  const int e0 = tid * per;
  const int e1 = (int64_t)(e0 + per) < len ? e0 + per : (int)(len > e0 ? len : e0);

  if (active) {
    for (int64_t base = 0; base < len; base += (int64_t)kPer * kTopkThreads) {
      float v[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {  // all loads first: one round trip per kPer elements
        const int64_t e = base + u * kTopkThreads + tid;
        v[u] = e < len ? __ldcg(sc + s0 + e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int64_t e = base + u * kTopkThreads + tid;
        if (e < len) keys[e] = float_order_key(v[u]);
      }
    }
  }
  for (int i = tid; i < kHistBins; i += kTopkThreads) hist[i] = 0;
  __syncthreads();
  if (!p.hist_done) {
    // first-level histogram of the chunk, added into the row's
    if (active)
      for (int u = 0; u < per; ++u) {
        const int e = e0 + u;
        hist_add(hist, e < e1, e < e1 ? keys[e] >> (32 - kHistBits) : 0u);
      }
    __syncthreads();
    for (int i = tid; i < kHistBins; i += kTopkThreads)
      if (hist[i]) atomicAdd(p.ghist + row * kHistBins + i, hist[i]), hist[i] = 0;
    if (!grid_barrier(p.gsync, ++nbar * nblk, p.dev_status, 40, p.wait_cycles)) return;
  }

  // phase 1: first-level threshold bin b1.  The chunk's keys in b1 (candidates) go to the
  // row's candidate list, one contiguous range per CTA in entry order, and are histogrammed
  // on their next 12 bits (needed only if some row's list overflows).
  uint32_t b1 = 0, above1 = 0;
  if (active) threshold_bin(p.ghist + row * kHistBins, (uint32_t)p.k, S, b1, above1);
  const uint32_t r = (uint32_t)p.k - above1;  // keys of bin b1 to keep (>= 1)
  uint32_t n_c = 0, n_s1 = 0;                 // this thread's candidates and keys above b1
  if (active)
    for (int u = 0; u < per; ++u) {
      const int e = e0 + u;
      const uint32_t key = e < e1 ? keys[e] : 0u;
      const uint32_t bin = key >> (32 - kHistBits);
      const bool c = e < e1 && bin == b1;
      n_c += c, n_s1 += (e < e1 && bin > b1);
      hist_add(hist, c, (key >> (32 - 2 * kHistBits)) & (kHistBins - 1));
    }
  uint32_t cb, z0, ctot, s1tot;
  block_scan_counts(n_c, n_s1, S, cb, z0, ctot, s1tot);  // (its barriers also complete the histogram)
  if (active) {
    // this CTA's candidates, in entry order, in its own region of the row's list
    uint2* mine = p.cand + ((int64_t)row * parts + part) * p.chunk;
    uint32_t x = cb;
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = keys[e];
      if ((key >> (32 - kHistBits)) == b1) mine[x++] = make_uint2(key, (uint32_t)(s0 + e));
    }
    if (tid == 0) {
      myslot[4] = (int32_t)s1tot, myslot[5] = (int32_t)ctot;
      if (ctot) atomicAdd(p.ncand + row, ctot);  // the row's total (no return value needed)
    }
  }
  for (int i = tid; i < kHistBins; i += kTopkThreads)
    if (hist[i]) atomicAdd(p.ghist2 + row * kHistBins + i, hist[i]);
  if (!grid_barrier(p.gsync, ++nbar * nblk, p.dev_status, 41, p.wait_cycles)) return;
  {
    // every CTA of the row has read the first-level histogram: clear this CTA's slice of it
    const int slice = (kHistBins + parts - 1) / parts;
    const int lo = part * slice, hi = lo + slice < kHistBins ? lo + slice : kHistBins;
    for (int i = lo + tid; i < hi; i += kTopkThreads) p.ghist[row * kHistBins + i] = 0u;
  }

  // phase 2 (rows with at most kCandListCap candidates): every CTA gathers the row's
  // candidates in entry order (CTA by CTA, at the prefix of the counts before it), finds
  // the second-level bin b2 from the row's second histogram, keeps the candidates whose
  // next 12 bits are above b2 and the r2 best (key desc, entry asc) of the few equal to
  // it, then writes its own kept entries at the offset given by the CTAs before it.
  __shared__ uint32_t p_pre[kNumSMs + 1];
  __shared__ int64_t s_sure;
  __shared__ uint32_t s_flags;  // bit 0: some row has more candidates than the cap
  uint32_t n_cand = 0;
  {
    // the per-CTA counts of this row (warp 0) and every row's total (warp 1), read
    // together with the second histogram below
    uint32_t cnt[5] = {0u, 0u, 0u, 0u, 0u};
    int64_t sure = 0;
    if (tid < 32 && active) {
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int q = tid * 5 + k;
        const int32_t* o = p.slots + ((int64_t)row * parts + q) * kGridSlot;
        if (q < parts) cnt[k] = (uint32_t)__ldcg(o + 5);
        if (q < part) sure += __ldcg(o + 4);
      }
    }
    if (tid >= 32 && tid < 64) {
      uint32_t over = 0;
      for (int rr = tid - 32; rr < (int)gridDim.y; rr += 32) over |= __ldcg(p.ncand + rr) > (uint32_t)kCandListCap;
      over = __any_sync(0xffffffffu, over != 0);
      if (tid == 32) s_flags = over;
    }
    if (tid < 32 && active) {
      uint32_t sum = cnt[0] + cnt[1] + cnt[2] + cnt[3] + cnt[4];
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += u;
      }
      uint32_t run = incl - sum;
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int q = tid * 5 + k;
        if (q < parts) p_pre[q] = run;
        run += cnt[k];
      }
      if (tid == 31) p_pre[parts] = incl;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sure += __shfl_xor_sync(0xffffffffu, sure, o);
      if (tid == 0) s_sure = sure;
    }
  }
  uint32_t b2 = 0, above2 = 0;
  if (active) threshold_bin(p.ghist2 + row * kHistBins, r, S, b2, above2);
  __syncthreads();  // the tables above are written
  const bool any_overflow = s_flags != 0u;  // the same for every CTA
  if (active) n_cand = p_pre[parts];
  const bool listed = active && n_cand <= (uint32_t)kCandListCap;
  const uint32_t r2 = r - above2;  // keys with the top 24 bits (b1, b2) to keep (>= 1)
  const uint32_t pre24 = (b1 << kHistBits) | b2;
  if (listed) {
    for (int i = tid; i < kCandListCap / 32; i += kTopkThreads) kbits[i] = 0u;
    for (uint32_t x = tid; x < n_cand; x += kTopkThreads) {
      int lo = 0, hi = parts - 1;  // the CTA that holds candidate x: the last q with p_pre[q] <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p_pre[mid] <= x) lo = mid; else hi = mid - 1;
      }
      sorted[x] = __ldcg(p.cand + ((int64_t)row * parts + lo) * p.chunk + (x - p_pre[lo]));
    }
    __syncthreads();
    // the sub-candidates (top 24 bits = (b1, b2)) in entry order, and their ranks
    uint32_t sub_base = 0;
    for (uint32_t base = 0; base < n_cand; base += kTopkThreads) {
      const uint32_t x = base + tid;
      const uint32_t key = x < n_cand ? sorted[x].x : 0u;
      const bool above = x < n_cand && (key >> 8) > pre24, sub = x < n_cand && (key >> 8) == pre24;
      uint32_t ab, sb, at, st;
      block_scan2(above, sub, S, ab, sb, at, st);
      if (above) atomicOr(&kbits[x >> 5], 1u << (x & 31));
      if (sub && sub_base + sb < (uint32_t)kSubListCap) list[sub_base + sb] = make_uint2(key, x);
      sub_base += st;
    }
    __syncthreads();
    const uint32_t n_sub = sub_base;  // >= r2
    if (n_sub <= (uint32_t)kSubListCap) {
      if (tid < (int)n_sub) {
        const uint2 me = list[tid];
        uint32_t rank = 0;
        for (uint32_t y = 0; y < n_sub; ++y) {
          const uint2 o = list[y];
          rank += o.x > me.x || (o.x == me.x && o.y < me.y);
        }
        if (rank < r2) atomicOr(&kbits[me.y >> 5], 1u << (me.y & 31));
      }
    } else {
      // many equal 24-bit prefixes: exact selection over the row's candidates
      uint32_t T, ties;
      auto sub24 = [&](int64_t x) { return (sorted[x].x >> 8) == pre24 ? sorted[x].x : 0u; };
      radix_select(sub24, n_cand, r2, S, T, ties);
      uint32_t eq_base = 0;
      for (uint32_t base = 0; base < n_cand; base += kTopkThreads) {
        const uint32_t x = base + tid;
        const uint32_t key = x < n_cand ? sub24(x) : 0u;
        const bool gt = x < n_cand && key > T && key != 0u, eq = x < n_cand && key == T && key != 0u;
        uint32_t gb, eb, gtt, ett;
        block_scan2(gt, eq, S, gb, eb, gtt, ett);
        if (gt || (eq && eq_base + eb < ties)) atomicOr(&kbits[x >> 5], 1u << (x & 31));
        eq_base += ett;
      }
    }
    __syncthreads();
    // kept candidates of the CTAs before this one
    const uint32_t mine0 = p_pre[part];
    uint32_t kc = 0;
    for (uint32_t w = tid; w * 32 < mine0; w += kTopkThreads) {
      const uint32_t bits = kbits[w];
      const uint32_t lim = mine0 - w * 32;
      kc += __popc(lim >= 32 ? bits : (bits & ((1u << lim) - 1u)));
    }
    const int64_t before = s_sure + block_sum(kc, S);
    // this CTA's kept entries, in entry order
    auto kept = [&](uint32_t key, uint32_t ci) {
      const uint32_t bin = key >> (32 - kHistBits);
      return bin > b1 || (bin == b1 && ((kbits[(mine0 + ci) >> 5] >> ((mine0 + ci) & 31)) & 1u));
    };
    uint32_t mine = 0, ci = cb;
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = keys[e];
      mine += kept(key, ci);
      ci += (key >> (32 - kHistBits)) == b1;
    }
    uint32_t kb, zb, kt, zt;
    block_scan_counts(mine, 0u, S, kb, zb, kt, zt);
    int64_t slot = before + kb;
    ci = cb;
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = keys[e];
      if (kept(key, ci)) {
        out[slot] = (int32_t)(s0 + e);
        if (out_sc) out_sc[slot] = key_to_float(key);
        ++slot;
      }
      ci += (key >> (32 - kHistBits)) == b1;
    }
  }

  // rows whose candidate list overflowed (many keys share their top 12 bits): a
  // second 12-bit level, then a list of the few sub-candidates or, if that overflows
  // too, the last 8 bits and the ties through a prefix over the CTAs
  const bool slow_row = active && !listed;
  if (any_overflow) {
  // phase 2s: sure keeps counted, sub-candidates (top 24 bits = (b1, b2)) listed
  uint32_t sure = 0;
  if (slow_row)
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = keys[e], t24 = key >> 8;
      sure += t24 > pre24;
      if (t24 == pre24) {
        const uint32_t slot = atomicAdd(p.nsub + row, 1u);
        if (slot < (uint32_t)kSubListCap)
          p.sub[row * kSubListCap + slot] = make_uint2(key, (uint32_t)(s0 + e));
        else
          atomicOr(p.gsync + 1, 1u);
      }
    }
  sure = block_sum(sure, S);
  if (slow_row && tid == 0) myslot[0] = (int32_t)sure;
  if (!grid_barrier(p.gsync, ++nbar * nblk, p.dev_status, 42, p.wait_cycles)) return;

  // phase 3s: select among the sub-candidates and write this chunk's kept entries
  const uint32_t n_sub = slow_row ? __ldcg(p.nsub + row) : 0u;
  const bool fast = slow_row && n_sub <= (uint32_t)kSubListCap;
  const bool sub_overflow = __ldcg(p.gsync + 1) != 0u;  // the same for every CTA
  if (fast) {
    for (int i = tid; i < (int)(p.chunk / 32); i += kTopkThreads) selb[i] = 0u;
    if (tid < (int)n_sub) list[tid] = __ldcg(p.sub + row * kSubListCap + tid);
    if (tid < 32) {
      int64_t acc = 0;
      for (int i = tid; i < part; i += 32) acc += __ldcg(p.slots + ((int64_t)row * parts + i) * kGridSlot);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (tid == 0) s_before = acc;
    }
    __syncthreads();
    // rank each sub-candidate by (key desc, entry asc): the r2 best are kept
    bool sel = false;
    uint32_t sx = 0;
    if (tid < (int)n_sub) {
      const uint2 me = list[tid];
      sx = me.y;
      uint32_t rank = 0;
      for (uint32_t y = 0; y < n_sub; ++y) {
        const uint2 o = list[y];
        rank += o.x > me.x || (o.x == me.x && o.y < me.y);
      }
      sel = rank < r2;
      if (sel && sx >= (uint32_t)s0 && sx < (uint32_t)(s0 + len)) {
        const uint32_t e = sx - (uint32_t)s0;
        atomicOr(&selb[e >> 5], 1u << (e & 31));
      }
    }
    const int64_t sel_before = __syncthreads_count(sel && sx < (uint32_t)s0);
    const int64_t before = s_before + sel_before;
    uint32_t mine = 0;
    for (int e = e0; e < e1; ++e) {
      const uint32_t t24 = keys[e] >> 8;
      mine += t24 > pre24 || (t24 == pre24 && ((selb[e >> 5] >> (e & 31)) & 1u));
    }
    uint32_t kb, z0, kt, z1;
    block_scan_counts(mine, 0u, S, kb, z0, kt, z1);
    int64_t slot = before + kb;
    for (int e = e0; e < e1; ++e) {
      const uint32_t t24 = keys[e] >> 8;
      if (t24 > pre24 || (t24 == pre24 && ((selb[e >> 5] >> (e & 31)) & 1u))) {
        const int64_t s = s0 + e;
        out[slot] = (int32_t)s;
        if (out_sc) out_sc[slot] = __ldcg(sc + s);
        ++slot;
      }
    }
  }
  if (sub_overflow) {
    // exact k-th key from the last 8 bits; ties kept lowest entry first over the CTAs
    const bool slow = slow_row && !fast;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    if (slow)
      for (int u = 0; u < per; ++u) {
        const int e = e0 + u;
        const uint32_t key = e < e1 ? keys[e] : 0u;
        hist_add(hist, e < e1 && (key >> 8) == pre24, key & 255u);
      }
    __syncthreads();
    if (slow && tid < 256 && hist[tid]) atomicAdd(p.hist3 + row * 256 + tid, hist[tid]);
    if (!grid_barrier(p.gsync, ++nbar * nblk, p.dev_status, 43, p.wait_cycles)) return;
    uint32_t T = 0, r3 = 0;
    if (slow) {
      if (tid < 32) {
        // lane l covers digits 255-8l .. 248-8l
        const int hi = 255 - 8 * tid;
        uint32_t c[8], lsum = 0;
#pragma unroll
        for (int d = 0; d < 8; ++d) c[d] = __ldcg(p.hist3 + row * 256 + hi - d), lsum += c[d];
        uint32_t incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += u;
        }
        const uint32_t excl = incl - lsum;
        if (excl < r2 && r2 <= incl) {
          uint32_t cum = excl;
          for (int d = 0; d < 8; ++d) {
            if (cum + c[d] >= r2) {
              S.prefix = (uint32_t)(hi - d);
              S.desired = r2 - cum;
              break;
            }
            cum += c[d];
          }
        }
      }
      __syncthreads();
      T = (pre24 << 8) | S.prefix;
      r3 = S.desired;  // keys equal to T to keep (>= 1)
    }
    uint32_t gt = 0, eq = 0;
    if (slow)
      for (int e = e0; e < e1; ++e) gt += keys[e] > T, eq += keys[e] == T;
    uint32_t gb, eb, gtot, etot;
    block_scan_counts(gt, eq, S, gb, eb, gtot, etot);
    if (slow && tid == 0) myslot[1] = (int32_t)gtot, myslot[2] = (int32_t)etot;
    if (!grid_barrier(p.gsync, ++nbar * nblk, p.dev_status, 44, p.wait_cycles)) return;
    if (slow) {
      if (tid < 32) {
        int64_t g_acc = 0, e_acc = 0;
        for (int i = tid; i < part; i += 32) {
          const int32_t* o = p.slots + ((int64_t)row * parts + i) * kGridSlot;
          g_acc += __ldcg(o + 1), e_acc += __ldcg(o + 2);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          g_acc += __shfl_xor_sync(0xffffffffu, g_acc, o);
          e_acc += __shfl_xor_sync(0xffffffffu, e_acc, o);
        }
        if (tid == 0) S.total = (uint32_t)e_acc, s_before = g_acc;
      }
      __syncthreads();
      const int64_t eq_before = S.total;
      const int64_t ties = r3 > eq_before ? std::min<int64_t>(r3 - eq_before, etot) : 0;  // ours to keep
      const int64_t base = s_before + std::min<int64_t>(r3, eq_before);
      int64_t g = gb, q = eb;
      for (int e = e0; e < e1; ++e) {
        const uint32_t key = keys[e];
        int64_t slot = -1;
        if (key > T) slot = g + std::min<int64_t>(q, ties), ++g;
        else if (key == T) slot = q < ties ? g + q : -1, ++q;
        if (slot >= 0) {
          const int64_t s = s0 + e;
          out[base + slot] = (int32_t)s;
          if (out_sc) out_sc[base + slot] = __ldcg(sc + s);
        }
      }
    }
  }
  }  // any_overflow
  if (!active) {
    for (int64_t i = (int64_t)part * kTopkThreads + tid; i < p.k; i += (int64_t)parts * kTopkThreads) {
      out[i] = i < vis ? (int32_t)i : -1;
      if (out_sc) out_sc[i] = i < vis ? __ldcg(sc + i) : -INFINITY;
    }
  }
  // Leave the counters zero for the next call: the row's last CTA to finish clears the
  // row's second-level histograms and list size, the grid's last the grid-wide words
  // (every CTA counts itself finished only after its last read of them).
  __shared__ int s_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(p.dep + row, 1u) == (uint32_t)(parts - 1);
  }
  __syncthreads();
  if (s_last) {
    for (int i = tid; i < kHistBins; i += kTopkThreads) p.ghist2[row * kHistBins + i] = 0u;
    for (int i = tid; i < 256; i += kTopkThreads) p.hist3[row * 256 + i] = 0u;
    if (tid == 0) p.nsub[row] = 0u, p.dep[row] = 0u;
  }
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.gsync + 2, 1u) == nblk - 1) {
      for (int rr = 0; rr < (int)gridDim.y; ++rr) p.ncand[rr] = 0u;
      p.gsync[0] = 0u, p.gsync[1] = 0u;
      __threadfence();
      p.gsync[2] = 0u;
    }
  }
}

// ------------------------------------------------------------------ host

struct TopkPlan {
  int kind;  // 0 = one stage, 1 = three kernels, 2 = grid
  int64_t chunk;
  int n_chunks;
};

static size_t grid_smem_bytes(int64_t chunk) {
  return (size_t)chunk * 4 + kHistBins * 4 + kSubListCap * 8 + (size_t)chunk / 8 + kCandListCap * 8 +
         kCandListCap / 8;
}

// One CTA of the grid plan fits an SM of the current device (cached per device).
static bool grid_plan_fits(int64_t chunk) {
  static int ok_dev[64] = {};  // 0 unknown, 1 fits, 2 does not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (ok_dev[dev] == 0) {
    int n = 0, sms = 0;
    const bool fits =
        cudaFuncSetAttribute(topk_grid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)grid_smem_bytes(kGridChunkCap)) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topk_grid_kernel, kTopkThreads,
                                                      grid_smem_bytes(kGridChunkCap)) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n >= 1 && sms >= kNumSMs;
    ok_dev[dev] = fits ? 1 : 2;
  }
  return chunk <= kGridChunkCap && ok_dev[dev] == 1;
}

static TopkPlan plan_topk(const hyb_index_args* a, int64_t n_vis_max) {
  TopkPlan pl{0, 0, 0};
  const int64_t rows = a->batch * a->n_q;
  // a short row stays on one CTA unless the rows are too few to fill the GPU (decode of a
  // few sequences): then the grid plan spreads each row over at least 8 SMs
  if (n_vis_max <= kStageCap && !(n_vis_max > kGridMinEntries && rows * 8 <= kNumSMs)) return pl;
  if (rows <= kNumSMs) {
    // grid plan: up to one CTA per SM, the row's entries split evenly
    const int64_t P = kNumSMs / rows;
    int64_t chunk = (n_vis_max + P - 1) / P;
    chunk = (chunk + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
    if (chunk <= kGridChunkCap && grid_plan_fits(chunk)) {
      pl.kind = 2;
      pl.chunk = chunk;
      pl.n_chunks = (int)((n_vis_max + chunk - 1) / chunk);
      return pl;
    }
  }
  int64_t P = (2 * kNumSMs + rows - 1) / rows;
  P = std::max<int64_t>(1, std::min<int64_t>(P, kMaxChunks));
  int64_t chunk = (n_vis_max + P - 1) / P;
  chunk = (chunk + 1023) / 1024 * 1024;
  pl.kind = 1;
  pl.chunk = chunk;
  pl.n_chunks = (int)((n_vis_max + chunk - 1) / chunk);
  return pl;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }


size_t topk_workspace_bytes(const hyb_index_args* a, int64_t n_vis_max) {
  const TopkPlan pl = plan_topk(a, n_vis_max);
  const size_t rows = (size_t)(a->batch * a->n_q);
  if (pl.kind == 2)
    return align256(rows * pl.n_chunks * kGridSlot * 4) + align256(rows * kSubListCap * 8) +
           align256(rows * pl.n_chunks * pl.chunk * 8);
  if (pl.kind != 1) return 0;
  const size_t region = rows * (size_t)pl.n_chunks * (size_t)pl.chunk;
  return align256(rows * kHistBins * 8 + rows * 4) + 3 * align256(region * 4) + align256(rows * pl.n_chunks * 8);
}

bool topk_shape_supported(const hyb_index_args* a, int64_t) { return a->k >= 1 && a->k <= 2048; }

static void topk_pointers(TopkParams& p, const TopkPlan& pl, int64_t rows, void* ws, void* zr) {
  char* w = static_cast<char*>(ws);
  if (pl.kind == 2) {
    // the counters (zero between calls) at fixed places of the workspace's start
    constexpr int64_t R = kNumSMs;
    p.ghist = static_cast<uint32_t*>(zr);
    p.ghist2 = p.ghist + R * kHistBins;
    p.hist3 = p.ghist2 + R * kHistBins;
    p.nsub = p.hist3 + R * 256;
    p.ncand = p.nsub + R;
    p.dep = p.ncand + R;
    p.gsync = p.dep + R;
    p.slots = reinterpret_cast<int32_t*>(w);
    w += align256((size_t)rows * pl.n_chunks * kGridSlot * 4);
    p.sub = reinterpret_cast<uint2*>(w);
    w += align256((size_t)rows * kSubListCap * 8);
    p.cand = reinterpret_cast<uint2*>(w);
    return;
  }
  const size_t region = (size_t)rows * pl.n_chunks * pl.chunk;
  p.ghist = reinterpret_cast<uint32_t*>(w);
  p.ghist2 = p.ghist + rows * kHistBins;
  p.done = p.ghist2 + rows * kHistBins;
  w += align256((size_t)rows * kHistBins * 8 + (size_t)rows * 4);
  p.def_idx = reinterpret_cast<int32_t*>(w);
  w += align256(region * 4);
  p.cand_key = reinterpret_cast<uint32_t*>(w);
  w += align256(region * 4);
  p.cand_idx = reinterpret_cast<int32_t*>(w);
  w += align256(region * 4);
  p.counts = reinterpret_cast<int32_t*>(w);
}

uint32_t* topk_prepare_hist(const hyb_index_args* a, int64_t n_vis_max, void* ws, void* zr, cudaStream_t s,
                            cudaError_t* err) {
  *err = cudaSuccess;
  const int64_t rows = a->batch * a->n_q;
  const TopkPlan pl = plan_topk(a, n_vis_max);
  if (rows == 0 || pl.kind == 0) return nullptr;
  TopkParams p{};
  topk_pointers(p, pl, rows, ws, zr);
  // the grid plan's counters are already zero (left so by the previous call); the
  // three-kernel plan clears its own
  if (pl.kind == 1) *err = cudaMemsetAsync(p.ghist, 0, (size_t)rows * (kHistBins * 8 + 4), s);
  return p.ghist;
}

cudaError_t launch_topk(const hyb_index_args* a, const float* scores, int64_t score_stride, void* ws, void* zr,
                        bool hist_done, cudaStream_t s) {
  TopkParams p{};
  p.scores = scores, p.score_stride = score_stride, p.idx = a->idx, p.out_scores = a->scores;
  p.n_q = a->n_q, p.n_entries = a->n_entries, p.m = a->m, p.k = a->k, p.q_pos0 = a->q_pos0, p.q_pos = a->q_pos;
  p.dev_status = a->dev_status;
  p.wait_cycles = grid_wait_cycles();
  const int64_t rows = a->batch * a->n_q;
  if (rows == 0) return cudaSuccess;
  const int64_t n_vis_max = a->q_pos ? a->n_entries
                                     : std::min<int64_t>(visible_entries(a->q_pos0 + a->n_q - 1, a->m), a->n_entries);
  const TopkPlan pl = plan_topk(a, n_vis_max);
  cudaError_t e;
  if (pl.kind == 0) {
    const size_t smem = sizeof(uint32_t) * (size_t)kStageCap;
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = launch_pdl(topk_row_kernel, dim3((unsigned)rows), dim3(kTopkThreads), smem, s, p)) != cudaSuccess)
      return e;
    return cudaGetLastError();
  }
  p.chunk = pl.chunk, p.n_chunks = pl.n_chunks;
  p.hist_done = hist_done ? 1 : 0;
  topk_pointers(p, pl, rows, ws, zr);
  const dim3 grid((unsigned)pl.n_chunks, (unsigned)rows);
  if (pl.kind == 2) {
    const size_t smem = grid_smem_bytes(pl.chunk);
    e = cudaFuncSetAttribute(topk_grid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // The kernel has grid-wide barriers, so every CTA must become resident: at most one
    // CTA per SM is launched and one CTA fits an SM (checked by the plan), so CTAs that
    // find their SM busy with other work start as that work drains.  (A cooperative launch
    // would state the same guarantee, but inside a CUDA graph next to copies it measured
    // slower.)  A permanent shortage of SMs ends as HYB_DEV_TIMEOUT from the bounded barrier.
    if ((e = launch_pdl(topk_grid_kernel, grid, dim3(kTopkThreads), smem, s, p)) != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (!hist_done) {  // the histograms were zeroed by topk_prepare_hist
    if ((e = launch_pdl(topk_hist_kernel, grid, dim3(kTopkThreads), 0, s, p)) != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t smem = (size_t)2 * a->k * 4 + (size_t)kSubCap * 8 + (size_t)kCandCap / 8;
  e = cudaFuncSetAttribute(topk_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(topk_filter_kernel, grid, dim3(kTopkThreads), smem, s, p)) != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hyb
