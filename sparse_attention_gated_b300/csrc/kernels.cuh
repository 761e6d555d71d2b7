// kernels.cuh -- launchers of the hybrid-attention kernels (internal to the
// library; the public boundary is include/hyb.h).  Arguments have already
// been validated by the C-ABI layer when these are called.
#pragma once

#include "common.cuh"

namespace hyb {

// Attention workspaces start with this many bytes of join counters, which must be zero
// before the first call and which every call leaves zero again.
constexpr size_t kJoinRegionBytes = 1024;

// top-k threshold histogram over the top bits of the order-preserving score keys
constexpr int kTopkHistBits = 12;
constexpr int kTopkHistBins = 1 << kTopkHistBits;
// The csa_index_topk workspace starts with the counters of the top-k grid plan (up to one
// row per SM): two histograms and a 256-bin one per row, three words per row, four for
// the grid.  They must be zero before the first call and every call leaves them zero.
constexpr size_t kTopkZeroRegionBytes =
    ((size_t)kNumSMs * (2 * kTopkHistBins + 256 + 3) * 4 + 4 * 4 + 255) / 256 * 256;

// Bound, in SM clock cycles, of the device-side waits that span CTAs (the top-k grid
// plan's grid barriers, the split joins of the attention kernel): the value set by
// hyb_set_grid_wait_limit, about 1 s by default.
constexpr long long kDefaultGridWaitCycles = 1LL << 31;
long long grid_wait_cycles();

// compress.cu
bool compress_shape_supported(int64_t c);
cudaError_t launch_compress(const hyb_compress_args* a, int64_t n_out, cudaStream_t s);
constexpr int kCompressBatchMax = 4;
// Several compressions in one launch (n <= kCompressBatchMax, one input type).
cudaError_t launch_compress_batch(const hyb_compress_args* const* a, const int64_t* n_out, int n, cudaStream_t s);

// norm_rope.cu
cudaError_t launch_norm_rope(const hyb_norm_rope_args* a, cudaStream_t s);
constexpr int kNormRopeBatchMax = 4;
cudaError_t launch_norm_rope_batch(const hyb_norm_rope_args* calls, int n, cudaStream_t s);

// out_proj.cu (tcgen05 grouped output projection: bf16 in, F32 or BF16 out)
bool out_proj_shape_supported(int64_t n_h, int64_t c, int64_t g, int64_t d_g);
cudaError_t launch_out_proj(const void* o, const void* w, void* out, int out_bf16, int64_t rows, int64_t n_h, int64_t c,
                            int64_t g, int64_t d_g, int64_t out_stride, int32_t* dev_status, cudaStream_t s);

// sink.cu: rows = batch * n_q * n_h rows of c values (out_dtype F32 or BF16) and their lse
cudaError_t launch_sink(void* out, int32_t out_dtype, float* lse, const float* sink, int64_t rows, int64_t n_h,
                        int64_t c, cudaStream_t s);

// indexer.cu (CUDA-core scores, any supported dtype)
bool index_cc_shape_supported(int64_t n_ih, int64_t c_I);
cudaError_t launch_index_scores_cc(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                   cudaStream_t s);

// indexer_tc.cu (tcgen05 FP8 scores: E4M3, c_I = 128, 64 indexer heads)
bool index_tc_shape_supported(const hyb_index_args* a);
// ghist (optional): the row histograms of the top-k plan; *hist_done tells whether this launch filled them
cudaError_t launch_index_scores_tc(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                   uint32_t* ghist, bool* hist_done, cudaStream_t s);
// MXFP4 scores (packed e2m1 keys and queries with e8m0 block scales) on the tensor cores
bool index_fp4_shape_supported(const hyb_index_args* a);
cudaError_t launch_index_scores_fp4(const hyb_index_args* a, float* scores, int64_t score_stride, int64_t n_vis_max,
                                    uint32_t* ghist, bool* hist_done, cudaStream_t s);

// topk.cu
// ws: the plan's scratch; zr: the zeroed counters (kTopkZeroRegionBytes at the workspace start)
size_t topk_workspace_bytes(const hyb_index_args* a, int64_t n_vis_max);
bool topk_shape_supported(const hyb_index_args* a, int64_t n_vis_max);
// the zeroed row histograms when the top-k plan uses them (else nullptr)
uint32_t* topk_prepare_hist(const hyb_index_args* a, int64_t n_vis_max, void* ws, void* zr, cudaStream_t s,
                            cudaError_t* err);
cudaError_t launch_topk(const hyb_index_args* a, const float* scores, int64_t score_stride, void* ws, void* zr,
                        bool hist_done, cudaStream_t s);

// attend_cc.cu (CUDA-core attention for all three entry sources)
struct AttendJob {
  int mode;  // 0 = CSA index list, 1 = HCA visible range, 2 = sliding window + merge
  const void* q;
  const void* k;
  const void* v;
  const int32_t* idx;
  float* o;
  float* lse;
  const float* o_in;
  const float* lse_in;
  void* out;
  int out_bf16;
  int64_t batch, n_q, n_h, c, n_entries, kv_stride, list_len, m, q_pos0, kv_pos0, n_win;
  float scale;
  int dtype;
  int32_t* dev_status;
  // modes 0/1: fused window merge (see hyb_window): raw rows wk [batch][w_stride][c] at
  // absolute positions w_pos0.., query 0 at wq_pos0; out / out_bf16 / n_win as in mode 2;
  // lse then receives the union's lse and o is not written
  int win;
  const void* wk;
  int64_t w_stride, w_pos0, wq_pos0;
  // optional device-side positions: q_pos [batch * n_q] absolute query positions (modes 1
  // and 2; NULL = q_pos0 + j), kv_pos0s [batch] per-sequence kv_pos0 of the window rows
  // (mode 2; NULL = kv_pos0); the fused window's own: wq_pos, w_pos0s
  const int64_t* q_pos;
  const int64_t* kv_pos0s;
  const int64_t* wq_pos;
  const int64_t* w_pos0s;
  // optional per-head sink logits [n_h] joined to the final result by the kernels that
  // write it (the 128-head kernel); NULL = none
  const float* sink;
};
bool attend_cc_shape_supported(int64_t c, int64_t n_h);

// attend_tc.cu (tcgen05 MQA attention: bf16, c = 512, heads in groups of 64)
bool attend_tc_supported(const AttendJob& j);
int attend_tc_splits(const AttendJob& j);
size_t attend_tc_workspace_bytes(const AttendJob& j);
cudaError_t launch_attend_tc(const AttendJob& j, void* ws, cudaStream_t s);
// attend_h128.cu (tcgen05 MQA attention with 128 heads per CTA: bf16, c = 512, key = value,
// lists and visible ranges of decode-shaped launches, window fused)
bool attend_h128_enabled();
bool attend_h128_supported(const AttendJob& j);
int attend_h128_splits(const AttendJob& j);
size_t attend_h128_workspace_bytes(const AttendJob& j);
cudaError_t launch_attend_h128(const AttendJob& j, void* ws, cudaStream_t s);
int attend_cc_splits(const AttendJob& j);
size_t attend_cc_workspace_bytes(const AttendJob& j);
cudaError_t launch_attend_cc(const AttendJob& j, void* ws, cudaStream_t s);

}  // namespace hyb
