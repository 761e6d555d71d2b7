/*
 * hyb.h -- C ABI of the B300 (sm_103a) hybrid-attention library: the
 * DeepSeek-V4 CSA / HCA / sliding-window attention forward.
 *
 * Sources (web pages on DeepSeek-V4, cited by title and section):
 *   [HA]  "DeepSeek-V4 hybrid attention: CSA, HCA, mHC, MoE" (trishampatil.com):
 *         V.1 compression with overlap, V.2 lightning indexer, V.3 core
 *         attention, VI heavily compressed attention.
 *   [DV4] "DeepSeek-V4: Anatomy of an Open-Source Frontier Model"
 *         (modernaiengineering.com): "One query in a CSA layer" steps 1-5.
 *   [KE]  "DeepSeek-V4 Architecture From Kernels" (shivasnotes.com):
 *         section 6 (the CSA attention contract: caller-owned buffers,
 *         explicit sizes and scale, an int index array), section 9
 *         (heterogeneous KV cache: tails, exact recent window).
 *   [MA]  "Mastering DeepSeek-V4 Architecture, Course 1" (mailtotanvir.github.io):
 *         model configurations table (m = 4, m' = 128, top-k, c = 512, c_I = 128).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers, row-major, innermost dimension
 *    last, densely packed unless a stride field says otherwise.  The caller
 *    allocates and frees all of them; the library keeps no pointer after the
 *    call returns and allocates no device memory.
 *  - Each call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronises the device.
 *  - Scratch memory: `workspace` must hold hyb_<call>_workspace_size(args)
 *    bytes (256-byte aligned device memory), or may be NULL when that size is
 *    0.  The workspace's contents need not be initialised.
 *  - Query positions: query j of every batch element sits at absolute token
 *    position t = q_pos0 + j (queries are consecutive positions), unless the
 *    call is given per-query positions: an optional `q_pos` array, int64
 *    [batch][n_q] in device memory, holding each query's own absolute position
 *    (a batch of sequences at different lengths, [KE] section 9's per-request
 *    cache).  The host cannot read those: a position that is negative, or that
 *    would see more compressed entries than exist or window rows outside the
 *    buffer, is clipped to what exists and reported as HYB_DEV_BAD_INDEX.
 *  - Visibility ([HA] V.2: only earlier blocks are scored; [KE] section 9): a compressed
 *    entry s built with compression factor m is visible to position t iff its
 *    last token is <= t, i.e. s < floor((t+1)/m).  Unfinished tails are covered
 *    by the sliding window.
 *  - Validation is host-side and happens before any launch; an invalid
 *    argument returns an error status and launches nothing.  Values that live
 *    in device memory (index lists) are range-checked by the kernels: a bad
 *    value is skipped and reported through the optional `dev_status` word
 *    (bits HYB_DEV_*), which the kernels only ever OR into.
 *  - Errors: HYB_ERR_INVALID_ARG (null pointer, bad size, misaligned pointer,
 *    inconsistent dtypes), HYB_ERR_UNSUPPORTED (a valid shape for which no
 *    kernel is compiled), HYB_ERR_WORKSPACE (workspace missing or too small),
 *    HYB_ERR_CUDA (a launch failed; hyb_last_error() holds the CUDA message).
 *    hyb_last_error() returns a thread-local description of the last failure.
 */
#ifndef HYB_H_
#define HYB_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HYB_API __attribute__((visibility("default")))
#else
#define HYB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hyb_status {
  HYB_OK = 0,
  HYB_ERR_INVALID_ARG = 1,
  HYB_ERR_UNSUPPORTED = 2,
  HYB_ERR_WORKSPACE = 3,
  HYB_ERR_CUDA = 4,
  HYB_ERR_TIMEOUT = 5
} hyb_status;

typedef enum hyb_dtype {
  HYB_F32 = 0,   /* IEEE binary32 */
  HYB_BF16 = 1,  /* bfloat16 (upper half of binary32) */
  HYB_E4M3 = 2,  /* OCP FP8 e4m3 (bias 7, max 448, no inf), one float32 scale per row */
  HYB_MXFP4 = 3  /* OCP microscaling FP4: e2m1 codes packed two per byte (element 2i in the
                    low nibble of byte i), one e8m0 scale byte (2^(e-127)) per block of 32
                    consecutive elements of a row */
} hyb_dtype;

/* bits OR-ed into *dev_status by the kernels */
#define HYB_DEV_BAD_INDEX 0x1 /* an index list held a value outside [-1, n_entries) */
#define HYB_DEV_TIMEOUT 0x2   /* a bounded device-side wait gave up */
/* bits 8-15 of *dev_status: with HYB_DEV_TIMEOUT, a nonzero kernel-internal
   identifier of the wait that gave up (diagnostic only) */
#define HYB_DEV_WAIT_SITE(status) (((status) >> 8) & 0xFF)

/* ------------------------------------------------------------------------
 * hyb_compress -- softmax-gated compressor ([HA] V.1 for CSA, [HA] VI for HCA;
 * [KE] section 6: a softmax over each block followed by a weighted sum).
 *
 * Pools each block of m consecutive token rows into one entry.  For entry i
 * and channel ch the gate is a softmax over the rows of its window of the
 * logits Z[row][ch] + bias[position][ch], and the entry is the gate-weighted
 * sum of C[row][ch]:
 *   overlap = 1 (CSA): window = stream b over block i-1 (positions 0..m-1)
 *                      followed by stream a over block i (positions m..2m-1);
 *                      one softmax over all 2m logits.  Block 0 has no block
 *                      -1: its stream-b logits are -inf.
 *   overlap = 0 (HCA): window = the m rows of block i (positions 0..m-1).
 *
 * Inputs ca, za (and cb, zb when overlap) are [batch][n_rows][c] of in_dtype
 * (F32 or BF16), sequence b starting in_batch_stride rows after sequence b-1
 * (0 means "= n_rows"; otherwise >= n_rows: the rows may be a window of a
 * longer per-sequence buffer); cb/zb must be NULL when overlap = 0.  bias is float32
 * [overlap ? 2m : m][c].  Row r of the inputs is absolute token
 * first_block*m + r; n_rows need not be a multiple of m (a trailing partial
 * block is a tail and produces nothing).
 *
 * Output: entries for the complete blocks, except that with overlap and
 * first_block > 0 the first block only serves as the previous block of the
 * next one (this is the decode-append form: pass the last 2m rows and
 * first_block = (t+1)/m - 2 to produce entry (t+1)/m - 1).  The count is
 * hyb_compress_out_count().  Output j is written at out + (b*out_batch_stride
 * + j)*c elements (out_batch_stride >= count; 0 means "= count"), of
 * out_dtype: F32, BF16 (round to nearest even) or E4M3 (per-entry scale
 * written to out_scale[b*out_batch_stride + j]: scale = amax/448 over the
 * entry's c channels, or 1 when amax = 0; code = nearest-even e4m3 of
 * value/scale, saturated to +-448; both divisions IEEE-rounded float32), or
 * MXFP4 (out: c/2 bytes per entry; out_scale, read as uint8*: c/32 e8m0 bytes
 * per entry at out_scale + (b*out_batch_stride + j)*(c/32); per block of 32
 * channels E = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 when amax
 * = 0), scale byte E + 127, code = nearest e2m1 of value * 2^-E, ties to the
 * even code, saturated to +-6; the decisions taken on the float32 result).
 * Arithmetic: float32 softmax and accumulation.
 * ------------------------------------------------------------------------ */
typedef struct hyb_compress_args {
  const void* ca;
  const void* cb;
  const void* za;
  const void* zb;
  const float* bias;
  void* out;
  float* out_scale;
  int64_t batch;
  int64_t n_rows;
  int64_t c;
  int64_t m;
  int64_t first_block;
  int64_t out_batch_stride;
  int64_t in_batch_stride; /* rows from one sequence's inputs to the next; 0 = n_rows */
  int32_t overlap;
  int32_t in_dtype;  /* hyb_dtype */
  int32_t out_dtype; /* hyb_dtype */
  int32_t* dev_status;
} hyb_compress_args;

HYB_API int64_t hyb_compress_out_count(int64_t n_rows, int64_t m, int32_t overlap, int64_t first_block);
HYB_API size_t hyb_compress_workspace_size(const hyb_compress_args* a);
HYB_API hyb_status hyb_compress(const hyb_compress_args* a, void* workspace, size_t ws_bytes, void* stream);

/* hyb_compress_batch -- up to HYB_COMPRESS_BATCH_MAX independent compressions in one launch:
 * each calls[i] computes exactly what hyb_compress(&calls[i], ...) computes (the entries
 * that complete at one decode step: the CSA entry, its indexer key and the HCA entry).
 * calls: host array of n_calls argument structs (read during the call only), all with the
 * same in_dtype; each is validated as hyb_compress validates it and nothing is launched if
 * one fails.  The calls must not write what another call reads.  No workspace. */
#define HYB_COMPRESS_BATCH_MAX 4
HYB_API hyb_status hyb_compress_batch(const hyb_compress_args* calls, int32_t n_calls, void* stream);

/* ------------------------------------------------------------------------
 * csa_index_topk -- lightning indexer scores and top-k selection
 * ([HA] V.2: I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . K_I[s]); keep the top-k;
 * [DV4] steps 2-3; the indexer runs at reduced precision).
 *
 * qI [batch][n_q][n_ih][c_I] and kI [batch][kv_stride][c_I] are both F32,
 * both E4M3 or both MXFP4 (dtype).  With E4M3 the decoded codes are
 * multiplied by qI_scale [batch][n_q][n_ih] and kI_scale [batch][kv_stride]
 * (float32); with MXFP4 qI and kI hold c_I/2 bytes per row and the scale
 * pointers, read as uint8*, hold c_I/32 e8m0 bytes per row (qI_scale
 * [batch][n_q][n_ih][c_I/32], kI_scale [batch][kv_stride][c_I/32]): each
 * element decodes to its e2m1 value times its block's 2^(e-127) (MXFP4 runs
 * on the tensor cores only: n_ih = 64, c_I = 128, kv_stride a multiple of 4);
 * with F32 both scale pointers must be NULL.  w [batch][n_q][n_ih] float32.
 * Entries 0..n_entries-1 exist; query j (position t = q_pos0 + j) scores only
 * the visible ones, s < floor((t+1)/m), and floor((q_pos0+n_q)/m) must not
 * exceed n_entries.
 *
 * Output idx [batch][n_q][k] int32: the min(k, visible) entries ranked first
 * by (score descending, entry index ascending), written in ascending entry
 * order and padded with -1.  Optional scores [batch][n_q][k] float32 receive
 * the selected entries' scores in the same order (-inf for padding).
 * Arithmetic: E4M3 products accumulated in float32 (tensor cores on
 * sm_103a), float32 ReLU and head reduction; the ranking compares the float32
 * scores exactly.
 * ------------------------------------------------------------------------ */
typedef struct hyb_index_args {
  const void* qI;
  const float* qI_scale;
  const float* w;
  const void* kI;
  const float* kI_scale;
  int32_t* idx;
  float* scores;
  int64_t batch;
  int64_t n_q;
  int64_t n_entries;
  int64_t kv_stride; /* entries between batch elements of kI / kI_scale; 0 means n_entries */
  int64_t n_ih;
  int64_t c_I;
  int64_t m;
  int64_t k;
  int64_t q_pos0;
  int32_t dtype; /* hyb_dtype: HYB_F32, HYB_E4M3 or HYB_MXFP4 */
  int32_t* dev_status;
  /* Optional profiling events (cudaEvent_t, or NULL): recorded on the stream
     right before and right after the scoring kernel, so that a caller can time
     the scoring apart from the selection.  While the stream is being captured
     into a graph they are recorded as external events (cudaEventRecordExternal),
     so they stay in the graph; otherwise they are recorded plainly.  The
     library neither creates nor destroys them. */
  void* ev_scores_begin;
  void* ev_scores_end;
  /* Optional per-query absolute positions, int64 [batch][n_q] in device memory
     (NULL: query j is at q_pos0 + j, and q_pos0 is ignored otherwise).  With them
     the workspace is sized for every row seeing all n_entries entries. */
  const int64_t* q_pos;
} hyb_index_args;

/* Workspace: csa_index_topk_workspace_size(a) bytes, 256-byte aligned.  Its
   first csa_index_topk_counter_bytes() bytes hold the top-k plan's counters
   (histograms, list sizes, a grid barrier), which must be zero before the
   first call that uses the workspace; every call leaves them zero again (the
   rest is scratch), so a caller zero-fills a workspace once, when it allocates
   it.  After a call that reported HYB_DEV_TIMEOUT, zero-fill those bytes again.
   csa_index_topk_counter_bytes() is a constant of the library build. */
HYB_API size_t csa_index_topk_workspace_size(const hyb_index_args* a);
HYB_API size_t csa_index_topk_counter_bytes(void);
HYB_API hyb_status csa_index_topk(const hyb_index_args* a, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * csa_index_topk_noalloc -- csa_index_topk for callers that cannot allocate
 * device memory.  (The method's description has no counterpart: this is a
 * deployment variant of the same computation.)
 *
 * Some callers cannot call cudaMalloc or a framework allocator at the point
 * where they run the indexer: code that owns no allocator (a plug-in inside a
 * host engine that hands it only input and output buffers), code that runs
 * under a fixed memory budget reserved up front, or code that must not touch
 * the allocator while it runs.  This entry point takes the same arguments as
 * csa_index_topk, but no workspace: its scratch is one file-scope device array
 * of HYB_NOALLOC_SCRATCH_BYTES, part of the library's image, which every GPU
 * that loads the library holds until the process exits.  The caller still
 * passes all inputs and outputs.
 *
 *  - The first call on a device looks up the array's device address (with that
 *    device current) and remembers it; make that first call before any stream
 *    capture.  Later calls allocate nothing and call no allocating routine.
 *  - Arguments needing more scratch than HYB_NOALLOC_SCRATCH_BYTES
 *    (csa_index_topk_workspace_size(a) > HYB_NOALLOC_SCRATCH_BYTES) are
 *    rejected with HYB_ERR_WORKSPACE before any launch.
 *  - Every call shares the one array, which keeps the previous call's
 *    contents: it starts zero-filled and every call leaves the counters that
 *    must start at zero zero again.  Calls whose work overlaps on the GPU
 *    (other streams, other host threads) race on it: serialise them on one
 *    stream.
 * ------------------------------------------------------------------------ */
#define HYB_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
HYB_API hyb_status csa_index_topk_noalloc(const hyb_index_args* a, void* stream);

/* csa_index_topk_noalloc_reset -- zero the counters at the start of the
 * library's scratch array on the current device, asynchronously on `stream`
 * (a memset of memory the library already holds: nothing is allocated).  A
 * call of csa_index_topk_noalloc that reported HYB_DEV_TIMEOUT can leave those
 * counters non-zero, and every later call on that device would then start
 * from them; call this once after such a call, before the next one (ordered
 * with it on the same stream).  Like csa_index_topk_noalloc, the first use on
 * a device looks up the array's address: make it before any stream capture. */
HYB_API hyb_status csa_index_topk_noalloc_reset(void* stream);

/* ------------------------------------------------------------------------
 * hyb_window -- the sliding-window branch fused into csa_attend / hca_attend.
 *
 * When the `window` member of their argument struct is not NULL, the call
 * returns what swa_merge returns for the compressed branch's result (swa_merge
 * with kw = vw = window->kw and o_in, lse_in = that result): `out` receives the
 * merged output and `lse` the log-sum-exp of the union; `o` is not written and
 * may be NULL.  Query j is at absolute position q_pos0 + j (for hca_attend it
 * must equal the call's q_pos0).  kw [batch][n_kv][c] (the call's dtype) holds
 * raw rows at absolute positions kv_pos0 ..; the window rows are both keys and
 * values, and every needed row must lie inside the buffer.  out
 * [batch][n_q][n_h][c] of out_dtype (F32 or BF16).  Where the launch fits the
 * GPU at once, the window is one more split of the compressed list's softmax
 * (no second kernel and no float32 o / lse round trip through memory);
 * otherwise the call runs the two steps in sequence.  (A fusion of two of the
 * method's steps for deployment; the result is the same.)
 * ------------------------------------------------------------------------ */
typedef struct hyb_window {
  const void* kw;
  int64_t n_kv;
  int64_t kv_pos0;
  int64_t q_pos0;
  int64_t n_win;
  void* out;
  int32_t out_dtype;
  /* Optional, device memory: q_pos int64 [batch][n_q] per-query positions (NULL:
     q_pos0 + j; for hca_attend they must be the call's own q_pos), kv_pos0s int64
     [batch] the absolute position of row 0 of each sequence's rows of kw (NULL:
     kv_pos0 for all), e.g. a per-sequence ring of raw rows. */
  const int64_t* q_pos;
  const int64_t* kv_pos0s;
} hyb_window;

/* ------------------------------------------------------------------------
 * csa_attend -- CSA core attention over the selected entries ([HA] V.3, MQA:
 * every head shares one compressed K and V; [KE] section 6 contract).
 *
 * For every head h of query (b, j):  p = softmax over the listed entries of
 * scale * q[b][j][h] . kc[b][s];  o[b][j][h] = sum p * vc[b][s];
 * lse[b][j][h] = natural log of the softmax denominator of the scaled scores.
 * idx [batch][n_q][k] int32 lists the entries; -1 entries are padding.  An
 * empty list gives o = 0 and lse = -inf.  q [batch][n_q][n_h][c]; kc, vc
 * [batch][kv_stride][c] (vc may equal kc: in the method key = value = the
 * compressed entries).  o float32 [batch][n_q][n_h][c], lse float32
 * [batch][n_q][n_h].  dtype F32 or BF16 (q, kc, vc); float32 accumulation.
 *
 * Optional attention sink ([HA] section IV: a learnable sink per head inside
 * both branches): with `sink` non-NULL (float32 [n_h], natural-log units) each
 * head's softmax denominator gains exp(sink[h]) with no value, once, on the
 * call's final result: o (or the fused window's out) is scaled by
 * exp(lse - L) and lse becomes L = log(exp(lse) + exp(sink[h])).  Because the
 * result is a log-sum-exp union, a later swa_merge of (o, lse) still yields
 * the sink applied to the whole union.
 * ------------------------------------------------------------------------ */
typedef struct hyb_csa_attend_args {
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* idx;
  float* o;
  float* lse;
  int64_t batch;
  int64_t n_q;
  int64_t n_h;
  int64_t c;
  int64_t n_entries;
  int64_t kv_stride; /* rows between batch elements of kc / vc; 0 means n_entries */
  int64_t k;
  float scale;
  int32_t dtype; /* hyb_dtype */
  int32_t* dev_status;
  const hyb_window* window; /* optional fused window merge (see hyb_window), or NULL */
  const float* sink;        /* optional per-head attention-sink logits [n_h], or NULL */
} hyb_csa_attend_args;

/* Workspace of csa_attend and hca_attend: *_workspace_size(a) bytes, 256-byte
   aligned.  Its first 1024 bytes hold counters that must be zero before the
   first call that uses the workspace; every call leaves them zero again (the
   rest is scratch), so a caller zero-fills a workspace once, when it allocates
   it.  After a call that reported HYB_DEV_TIMEOUT, zero-fill it again. */
HYB_API size_t csa_attend_workspace_size(const hyb_csa_attend_args* a);
HYB_API hyb_status csa_attend(const hyb_csa_attend_args* a, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * hca_attend -- HCA core attention, dense over every visible entry ([HA] VI).
 *
 * Like csa_attend, with the entry list of query j being 0 .. V-1,
 * V = floor((q_pos0 + j + 1)/m) (compression factor m of the HCA entries);
 * floor((q_pos0 + n_q)/m) must not exceed n_entries.
 * ------------------------------------------------------------------------ */
typedef struct hyb_hca_attend_args {
  const void* q;
  const void* kc;
  const void* vc;
  float* o;
  float* lse;
  int64_t batch;
  int64_t n_q;
  int64_t n_h;
  int64_t c;
  int64_t n_entries;
  int64_t kv_stride;
  int64_t m;
  int64_t q_pos0;
  float scale;
  int32_t dtype;
  int32_t* dev_status;
  const hyb_window* window; /* optional fused window merge (see hyb_window), or NULL */
  const float* sink;        /* optional per-head attention-sink logits [n_h], or NULL (see csa_attend) */
  const int64_t* q_pos;     /* optional per-query positions int64 [batch][n_q], device memory, or NULL */
} hyb_hca_attend_args;

HYB_API size_t hca_attend_workspace_size(const hyb_hca_attend_args* a);
HYB_API hyb_status hca_attend(const hyb_hca_attend_args* a, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * swa_merge -- sliding-window branch merged by log-sum-exp ([DV4] steps 4-5:
 * the last n_win uncompressed tokens and the compressed entries are attended
 * as one set; [KE] section 9: the most recent 128 tokens stay uncompressed).
 *
 * Query j at position t attends the raw rows at absolute positions
 * max(0, t-n_win+1) .. t, read from kw / vw [batch][n_kv][c] whose row 0 is
 * absolute position kv_pos0 (every needed row must lie inside the buffer).
 * The window result (o_w, lse_w) is merged with the compressed-branch result
 * (o_in float32 [batch][n_q][n_h][c], lse_in float32 [batch][n_q][n_h]):
 *   L = logaddexp(lse_in, lse_w);  out = e^(lse_in-L) o_in + e^(lse_w-L) o_w,
 * which equals one softmax over the union of both key sets.  o_in and lse_in
 * may both be NULL (no compressed branch).  out [batch][n_q][n_h][c] of
 * out_dtype (F32 or BF16); lse_out (optional, float32) receives L.
 * dtype (q, kw, vw): F32 or BF16.
 * ------------------------------------------------------------------------ */
typedef struct hyb_swa_args {
  const void* q;
  const void* kw;
  const void* vw;
  const float* o_in;
  const float* lse_in;
  void* out;
  float* lse_out;
  int64_t batch;
  int64_t n_q;
  int64_t n_h;
  int64_t c;
  int64_t n_kv;
  int64_t kv_pos0;
  int64_t q_pos0;
  int64_t n_win;
  float scale;
  int32_t dtype;
  int32_t out_dtype;
  int32_t* dev_status;
  const int64_t* q_pos;    /* optional per-query positions int64 [batch][n_q], device memory, or NULL */
  const int64_t* kv_pos0s; /* optional int64 [batch]: absolute position of row 0 of each sequence's kw / vw rows */
} hyb_swa_args;

HYB_API size_t swa_merge_workspace_size(const hyb_swa_args* a);
HYB_API hyb_status swa_merge(const hyb_swa_args* a, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * hyb_rmsnorm_rope -- RMSNorm of each row, then rotary encoding of the row's
 * last rope_dims dimensions ([HA] section IV: queries and compressed KV
 * entries are RMS-normalised inside both branches, and only their last 64
 * dimensions carry rotary position; rotary convention of [JH] "The Code: RoPE
 * Helpers": consecutive pairs, frequencies theta^(-2i/d)).
 *
 * In place on x [rows][c] of dtype F32 or BF16 (c even):
 *   y = x / sqrt(mean over the row of x^2 + eps) * gamma   (gamma float32 [c],
 *       NULL = ones; eps >= 0),
 *   then the pairs (2i, 2i+1) of the last rope_dims dimensions (even, <= c;
 *   0 = none) are rotated by the angle pos * theta^(-2i / rope_dims), pos =
 *   pos[r / rows_per_pos] (int64 absolute positions, rows_per_pos >= 1, e.g.
 *   n_h for a query's heads; NULL with rope_dims > 0 is an error).
 * Float32 arithmetic; the angle is formed and reduced in float64, so that
 * positions in the millions keep full float32 accuracy.  row_stride: elements
 * from one row to the next (0 = c; otherwise an even number >= c), so that one
 * call reaches strided rows such as one cache slot of every sequence.  No
 * workspace.
 * ------------------------------------------------------------------------ */
typedef struct hyb_norm_rope_args {
  void* x;
  int64_t rows;
  int64_t c;
  const float* gamma;
  float eps;
  int32_t dtype; /* hyb_dtype: F32 or BF16 */
  const int64_t* pos;
  int64_t rows_per_pos;
  int64_t rope_dims;
  double theta;
  int64_t row_stride;
} hyb_norm_rope_args;

HYB_API hyb_status hyb_rmsnorm_rope(const hyb_norm_rope_args* a, void* stream);

/* Up to HYB_NORM_ROPE_BATCH_MAX calls of one dtype in one launch (the queries and the
 * completed entries of a decode step's two layers, say): each call is validated as
 * hyb_rmsnorm_rope validates it, before anything is launched; the calls' rows must not
 * overlap.  n_calls 0 does nothing; calls are read on the host only. */
#define HYB_NORM_ROPE_BATCH_MAX 4
HYB_API hyb_status hyb_rmsnorm_rope_batch(const hyb_norm_rope_args* calls, int32_t n_calls, void* stream);

/* ------------------------------------------------------------------------
 * hyb_grouped_out_proj -- grouped output projection ([HA] section V.3, core
 * attention and grouped output: the n_h heads are split into g groups of
 * n_h/g consecutive heads, each group's (n_h/g)*c values are projected by a
 * matrix of its own, and the g results are concatenated; [MA] model
 * configurations table: g / d_g = 16 / 1024 (Pro), 8 / 1024 (Flash)).
 *
 *   out[r][j*d_g + e] = sum_k w[j][e][k] * o[r][j*(n_h/g)*c + k]
 *
 * o [rows][n_h][c] and w [g][d_g][(n_h/g)*c] are bf16 (dtype HYB_BF16); out
 * [rows][g*d_g] is F32 or BF16 (out_dtype); float32 accumulation on the
 * tensor cores.  g must divide n_h, d_g must be a multiple of 128 and
 * (n_h/g)*c a multiple of 64.  With g = 1 the call is a plain projection of
 * all n_h*c values (e.g. the concatenated g*d_g features mapped to the model
 * dimension: pass them as o [rows][1][g*d_g]).  out_row_stride: elements from
 * one output row to the next (0 = g*d_g; otherwise >= g*d_g), so that two
 * calls can fill the two halves of one output row (the projection of a
 * concatenation whose groups do not straddle it).  No workspace.  Pointers
 * 16-byte aligned.
 * ------------------------------------------------------------------------ */
typedef struct hyb_gproj_args {
  const void* o;
  const void* w;
  void* out;
  int64_t rows;
  int64_t n_h;
  int64_t c;
  int64_t g;
  int64_t d_g;
  int32_t dtype;     /* hyb_dtype of o and w: HYB_BF16 */
  int32_t out_dtype; /* hyb_dtype: HYB_F32 or HYB_BF16 */
  int32_t* dev_status;
  int64_t out_row_stride; /* 0 = g*d_g */
} hyb_gproj_args;

HYB_API hyb_status hyb_grouped_out_proj(const hyb_gproj_args* a, void* stream);

/* ------------------------------------------------------------------------
 * hyb_set_grid_wait_limit -- bound of the device-side waits that span CTAs.
 *
 * Two kernels wait on other CTAs of their grid: the top-k grid plan of
 * csa_index_topk (grid barriers between its phases) and the split join of the
 * tensor-core csa_attend / hca_attend (the splits of one query meet before
 * they merge).  Each such wait gives up after this many SM clock cycles; the
 * kernel then ORs HYB_DEV_TIMEOUT (and the wait's site in bits 8-15) into
 * dev_status and returns without hanging.  The default, about 1 s
 * (2^31 cycles), is reached only when CTAs of the launch cannot all become
 * resident (another context holding SMs).  A small limit makes such waits
 * expire on purpose, which is how failure detection is tested.  cycles < 0
 * restores the default.  Process-wide; applies to launches issued after the
 * call.  Returns the previous limit.  After a call that reported
 * HYB_DEV_TIMEOUT, the counters of its workspace must be zero-filled again
 * (see the workspace notes of csa_index_topk and csa_attend, and
 * csa_index_topk_noalloc_reset).  (Waits inside one CTA -- mbarriers of the
 * copy / tensor-core pipelines -- keep their fixed bound of about 1 s.)
 * ------------------------------------------------------------------------ */
HYB_API int64_t hyb_set_grid_wait_limit(int64_t cycles);

/* ------------------------------------------------------------------------ misc */
HYB_API const char* hyb_status_string(hyb_status s);
HYB_API const char* hyb_last_error(void);
/* Library version and the SM architecture the kernels were built for (1030 = sm_103a). */
HYB_API int32_t hyb_version(void);
HYB_API int32_t hyb_built_arch(void);

#ifdef __cplusplus
}
#endif

#endif /* HYB_H_ */
