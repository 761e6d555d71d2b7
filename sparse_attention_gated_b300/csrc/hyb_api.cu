// hyb_api.cu -- the C ABI declared in include/hyb.h: host-side argument
// validation (before any launch), workspace sizing, dispatch to the kernels
// and error reporting.  No device memory is allocated here.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "kernels.cuh"

#ifndef HYB_BUILT_ARCH
#define HYB_BUILT_ARCH 1030
#endif

namespace {

thread_local std::string g_last_error = "";

hyb_status fail(hyb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

hyb_status ok() {
  g_last_error.clear();
  return HYB_OK;
}

hyb_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(HYB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return a <= 1 || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(int32_t dt) { return dt == HYB_F32 ? 4 : dt == HYB_BF16 ? 2 : 1; }

// alignment a warp-lane vector access needs: V = c/32 elements, capped at 16 bytes
size_t lane_align(int64_t c, int32_t dt) {
  size_t bytes = (size_t)(c / 32) * elem_size(dt);
  return bytes >= 16 ? 16 : bytes;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A caller's profiling event: an external event node while the stream is being captured
// into a graph (so that it stays in the graph), a plain record otherwise.
cudaError_t record_event(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s,
                                  cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

int64_t n_vis_max(int64_t q_pos0, int64_t n_q, int64_t m, int64_t n_entries) {
  if (n_q <= 0) return 0;
  int64_t v = hyb::visible_entries(q_pos0 + n_q - 1, m);
  return v < n_entries ? v : n_entries;
}

// the most entries any query of an index call sees: with per-query positions in device
// memory the host cannot tell, so every row is sized for all of them
int64_t index_vis_max(const hyb_index_args* a) {
  if (a->n_q <= 0) return 0;
  return a->q_pos ? a->n_entries : n_vis_max(a->q_pos0, a->n_q, a->m, a->n_entries);
}

std::atomic<long long> g_grid_wait_cycles{hyb::kDefaultGridWaitCycles};

}  // namespace

long long hyb::grid_wait_cycles() { return g_grid_wait_cycles.load(std::memory_order_relaxed); }

extern "C" {

int32_t hyb_version(void) { return 1; }

int64_t hyb_set_grid_wait_limit(int64_t cycles) {
  return g_grid_wait_cycles.exchange(cycles < 0 ? hyb::kDefaultGridWaitCycles : (long long)cycles);
}
int32_t hyb_built_arch(void) { return HYB_BUILT_ARCH; }

const char* hyb_status_string(hyb_status s) {
  switch (s) {
    case HYB_OK: return "HYB_OK";
    case HYB_ERR_INVALID_ARG: return "HYB_ERR_INVALID_ARG";
    case HYB_ERR_UNSUPPORTED: return "HYB_ERR_UNSUPPORTED";
    case HYB_ERR_WORKSPACE: return "HYB_ERR_WORKSPACE";
    case HYB_ERR_CUDA: return "HYB_ERR_CUDA";
    case HYB_ERR_TIMEOUT: return "HYB_ERR_TIMEOUT";
  }
  return "HYB_ERR_UNKNOWN";
}

const char* hyb_last_error(void) { return g_last_error.c_str(); }

// ---------------------------------------------------------------- compress

int64_t hyb_compress_out_count(int64_t n_rows, int64_t m, int32_t overlap, int64_t first_block) {
  if (m <= 0 || n_rows < 0) return 0;
  const int64_t blocks = n_rows / m;
  const int64_t skip = (overlap && first_block > 0) ? 1 : 0;
  return blocks > skip ? blocks - skip : 0;
}

size_t hyb_compress_workspace_size(const hyb_compress_args*) { return 0; }

static hyb_status validate_compress(const hyb_compress_args* a, int64_t* n_out) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: args is NULL");
  if (a->batch < 0 || a->n_rows < 0 || a->m < 1 || a->first_block < 0 || a->out_batch_stride < 0 ||
      a->in_batch_stride < 0)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: negative size or m < 1");
  if (a->in_batch_stride != 0 && a->in_batch_stride < a->n_rows)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: in_batch_stride %lld < n_rows %lld", (long long)a->in_batch_stride,
                (long long)a->n_rows);
  if (a->overlap != 0 && a->overlap != 1) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: overlap must be 0 or 1");
  if (a->in_dtype != HYB_F32 && a->in_dtype != HYB_BF16)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: in_dtype must be F32 or BF16");
  if (a->out_dtype != HYB_F32 && a->out_dtype != HYB_BF16 && a->out_dtype != HYB_E4M3 && a->out_dtype != HYB_MXFP4)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: bad out_dtype");
  if (a->c < 1) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: c < 1");
  if (!hyb::compress_shape_supported(a->c))
    return fail(HYB_ERR_UNSUPPORTED, "hyb_compress: c = %lld not compiled (32, 64, 128, 256, 512)", (long long)a->c);
  *n_out = hyb_compress_out_count(a->n_rows, a->m, a->overlap, a->first_block);
  if (a->out_batch_stride != 0 && a->out_batch_stride < *n_out)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: out_batch_stride %lld < entries %lld",
                (long long)a->out_batch_stride, (long long)*n_out);
  if (!a->overlap && (a->cb || a->zb)) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: cb/zb must be NULL without overlap");
  if (*n_out == 0 || a->batch == 0) return ok();
  if (!a->ca || !a->za || !a->bias || !a->out) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: NULL ca/za/bias/out");
  if (a->overlap && (!a->cb || !a->zb)) return fail(HYB_ERR_INVALID_ARG, "hyb_compress: overlap needs cb and zb");
  const bool scaled = a->out_dtype == HYB_E4M3 || a->out_dtype == HYB_MXFP4;
  if (scaled != (a->out_scale != nullptr))
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: out_scale is required for E4M3 and MXFP4 output and only then");
  // the kernel moves 4 consecutive channels per access
  const size_t ai = 4 * elem_size(a->in_dtype);
  if (!aligned(a->ca, ai) || !aligned(a->za, ai) || (a->overlap && (!aligned(a->cb, ai) || !aligned(a->zb, ai))) ||
      !aligned(a->bias, 16) || !aligned(a->out, a->out_dtype == HYB_MXFP4 ? 2 : 4 * elem_size(a->out_dtype)) ||
      !aligned(a->out_scale, a->out_dtype == HYB_MXFP4 ? 1 : 4))
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress: misaligned pointer");
  return ok();
}

hyb_status hyb_compress(const hyb_compress_args* a, void*, size_t, void* stream) {
  int64_t n_out = 0;
  hyb_status st = validate_compress(a, &n_out);
  if (st != HYB_OK || n_out == 0 || a->batch == 0) return st;
  return cuda_status(hyb::launch_compress(a, n_out, static_cast<cudaStream_t>(stream)), "hyb_compress launch");
}

hyb_status hyb_compress_batch(const hyb_compress_args* calls, int32_t n_calls, void* stream) {
  static_assert(HYB_COMPRESS_BATCH_MAX == hyb::kCompressBatchMax, "batch size");
  if (n_calls < 0 || n_calls > HYB_COMPRESS_BATCH_MAX)
    return fail(HYB_ERR_INVALID_ARG, "hyb_compress_batch: n_calls = %d outside 0..%d", n_calls, HYB_COMPRESS_BATCH_MAX);
  if (n_calls > 0 && !calls) return fail(HYB_ERR_INVALID_ARG, "hyb_compress_batch: calls is NULL");
  const hyb_compress_args* ptr[HYB_COMPRESS_BATCH_MAX];
  int64_t n_out[HYB_COMPRESS_BATCH_MAX];
  for (int i = 0; i < n_calls; ++i) {
    hyb_status st = validate_compress(&calls[i], &n_out[i]);
    if (st != HYB_OK) return st;
    if (calls[i].in_dtype != calls[0].in_dtype)
      return fail(HYB_ERR_INVALID_ARG, "hyb_compress_batch: calls %d and 0 have different in_dtype", i);
    ptr[i] = &calls[i];
  }
  if (n_calls == 0) return ok();
  return cuda_status(hyb::launch_compress_batch(ptr, n_out, n_calls, static_cast<cudaStream_t>(stream)),
                     "hyb_compress_batch launch");
}

// ---------------------------------------------------------------- index + top-k

static size_t index_scores_bytes(const hyb_index_args* a) {
  const int64_t nv = index_vis_max(a);
  return round_up((size_t)(a->batch * a->n_q) * (size_t)nv * sizeof(float), 256);
}

size_t csa_index_topk_counter_bytes(void) { return hyb::kTopkZeroRegionBytes; }

size_t csa_index_topk_workspace_size(const hyb_index_args* a) {
  if (!a || a->batch <= 0 || a->n_q <= 0 || a->m < 1) return 0;
  const int64_t nv = index_vis_max(a);
  return hyb::kTopkZeroRegionBytes + index_scores_bytes(a) + round_up(hyb::topk_workspace_bytes(a, nv), 256);
}

static hyb_status validate_index(const hyb_index_args* a) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: args is NULL");
  if (a->batch < 0 || a->n_q < 0 || a->n_entries < 0 || a->kv_stride < 0 || a->q_pos0 < 0 || a->m < 1)
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: negative size or m < 1");
  if (a->dtype != HYB_F32 && a->dtype != HYB_E4M3 && a->dtype != HYB_MXFP4)
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: dtype must be F32, E4M3 or MXFP4");
  if (a->k < 1 || a->n_ih < 1 || a->c_I < 1) return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: k, n_ih, c_I must be >= 1");
  if (a->k > 2048) return fail(HYB_ERR_UNSUPPORTED, "csa_index_topk: k = %lld > 2048", (long long)a->k);
  if (!hyb::index_cc_shape_supported(a->n_ih, a->c_I))
    return fail(HYB_ERR_UNSUPPORTED, "csa_index_topk: n_ih = %lld / c_I = %lld not supported", (long long)a->n_ih,
                (long long)a->c_I);
  if (a->kv_stride != 0 && a->kv_stride < a->n_entries)
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: kv_stride < n_entries");
  if (!a->q_pos && a->n_q > 0 && hyb::visible_entries(a->q_pos0 + a->n_q - 1, a->m) > a->n_entries)
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: the last query sees %lld entries but only %lld exist",
                (long long)hyb::visible_entries(a->q_pos0 + a->n_q - 1, a->m), (long long)a->n_entries);
  if (a->batch == 0 || a->n_q == 0) return ok();
  if (!hyb::topk_shape_supported(a, index_vis_max(a)))
    return fail(HYB_ERR_UNSUPPORTED, "csa_index_topk: %lld visible entries with k = %lld exceed the top-k plan",
                (long long)index_vis_max(a), (long long)a->k);
  if (!a->qI || !a->w || !a->idx) return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: NULL qI/w/idx");
  if (a->n_entries > 0 && !a->kI) return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: NULL kI");
  const bool fp8 = a->dtype == HYB_E4M3 || a->dtype == HYB_MXFP4;
  if (fp8 && (!a->qI_scale || (a->n_entries > 0 && !a->kI_scale)))
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: E4M3 and MXFP4 need qI_scale and kI_scale");
  if (a->dtype == HYB_MXFP4 && !hyb::index_fp4_shape_supported(a))
    return fail(HYB_ERR_UNSUPPORTED, "csa_index_topk: MXFP4 runs with n_ih = 64, c_I = 128, kv_stride a multiple of 4 "
                "and 16-byte aligned qI, kI and scales only");
  if (!fp8 && (a->qI_scale || a->kI_scale))
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: scales must be NULL for F32");
  if (!aligned(a->kI, 16) || !aligned(a->qI, 4) || !aligned(a->w, 4) || !aligned(a->idx, 4) || !aligned(a->scores, 4) ||
      !aligned(a->q_pos, 8))
    return fail(HYB_ERR_INVALID_ARG, "csa_index_topk: misaligned pointer (kI needs 16 bytes, q_pos 8)");
  return ok();
}

hyb_status csa_index_topk(const hyb_index_args* a, void* workspace, size_t ws_bytes, void* stream) {
  hyb_status st = validate_index(a);
  if (st != HYB_OK || a->batch == 0 || a->n_q == 0) return st;
  const size_t need = csa_index_topk_workspace_size(a);
  if (need > 0 && (!workspace || ws_bytes < need))
    return fail(HYB_ERR_WORKSPACE, "csa_index_topk: workspace of %zu bytes needed, %zu given", need, ws_bytes);
  if (!aligned(workspace, 256)) return fail(HYB_ERR_WORKSPACE, "csa_index_topk: workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nv = index_vis_max(a);
  // [counters that stay zero between calls][scores][top-k scratch]
  void* zr = workspace;
  float* scores = reinterpret_cast<float*>(static_cast<char*>(workspace) + hyb::kTopkZeroRegionBytes);
  void* topk_ws = static_cast<char*>(workspace) + hyb::kTopkZeroRegionBytes + index_scores_bytes(a);
  cudaError_t e;
  uint32_t* ghist = hyb::topk_prepare_hist(a, nv, topk_ws, zr, s, &e);
  if (e != cudaSuccess) return cuda_status(e, "csa_index_topk: histogram reset");
  bool hist_done = false;
  if (a->ev_scores_begin && (e = record_event(a->ev_scores_begin, s)) != cudaSuccess)
    return cuda_status(e, "csa_index_topk: ev_scores_begin");
  e = a->dtype == HYB_MXFP4             ? hyb::launch_index_scores_fp4(a, scores, nv, nv, ghist, &hist_done, s)
      : hyb::index_tc_shape_supported(a) ? hyb::launch_index_scores_tc(a, scores, nv, nv, ghist, &hist_done, s)
                                         : hyb::launch_index_scores_cc(a, scores, nv, nv, s);
  if (e != cudaSuccess) return cuda_status(e, "csa_index_topk: index-score launch");
  if (a->ev_scores_end && (e = record_event(a->ev_scores_end, s)) != cudaSuccess)
    return cuda_status(e, "csa_index_topk: ev_scores_end");
  return cuda_status(hyb::launch_topk(a, scores, nv, topk_ws, zr, hist_done, s), "csa_index_topk: top-k launch");
}

// ----------------------------------------------- index + top-k, no allocation

namespace {

// The scratch of csa_index_topk_noalloc: part of the library image, held by every
// device that loads the library.  Host code never uses its name as an address: the
// device address comes from cudaGetSymbolAddress, once per device.
__device__ __align__(256) uint8_t g_noalloc_scratch[HYB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

// The device address of the scratch array on the current device, looked up once per
// device (with that device current) and remembered.
static hyb_status noalloc_scratch(const char* name, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, name);
  if (dev < 0 || dev >= kMaxDevices) return fail(HYB_ERR_UNSUPPORTED, "%s: device %d", name, dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e, name);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return HYB_OK;
}

hyb_status csa_index_topk_noalloc(const hyb_index_args* a, void* stream) {
  hyb_status st = validate_index(a);
  if (st != HYB_OK || a->batch == 0 || a->n_q == 0) return st;
  const size_t need = csa_index_topk_workspace_size(a);
  if (need > HYB_NOALLOC_SCRATCH_BYTES)
    return fail(HYB_ERR_WORKSPACE, "csa_index_topk_noalloc: these sizes need %zu bytes of scratch, more than the %zu "
                "bytes the library holds", need, (size_t)HYB_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if ((st = noalloc_scratch("csa_index_topk_noalloc", &scratch)) != HYB_OK) return st;
  return csa_index_topk(a, scratch, HYB_NOALLOC_SCRATCH_BYTES, stream);
}

hyb_status csa_index_topk_noalloc_reset(void* stream) {
  void* scratch = nullptr;
  hyb_status st = noalloc_scratch("csa_index_topk_noalloc_reset", &scratch);
  if (st != HYB_OK) return st;
  // a memset of memory the library already holds: nothing is allocated
  return cuda_status(cudaMemsetAsync(scratch, 0, hyb::kTopkZeroRegionBytes, static_cast<cudaStream_t>(stream)),
                     "csa_index_topk_noalloc_reset");
}

// ---------------------------------------------------------------- attention

static hyb::AttendJob csa_job(const hyb_csa_attend_args* a) {
  hyb::AttendJob j{};
  j.mode = 0, j.q = a->q, j.k = a->kc, j.v = a->vc, j.idx = a->idx, j.o = a->o, j.lse = a->lse;
  j.batch = a->batch, j.n_q = a->n_q, j.n_h = a->n_h, j.c = a->c, j.n_entries = a->n_entries;
  j.kv_stride = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  j.list_len = a->k, j.scale = a->scale, j.dtype = a->dtype, j.dev_status = a->dev_status;
  return j;
}

static hyb::AttendJob hca_job(const hyb_hca_attend_args* a) {
  hyb::AttendJob j{};
  j.mode = 1, j.q = a->q, j.k = a->kc, j.v = a->vc, j.o = a->o, j.lse = a->lse;
  j.batch = a->batch, j.n_q = a->n_q, j.n_h = a->n_h, j.c = a->c, j.n_entries = a->n_entries;
  j.kv_stride = a->kv_stride > 0 ? a->kv_stride : a->n_entries;
  j.m = a->m, j.q_pos0 = a->q_pos0, j.scale = a->scale, j.dtype = a->dtype, j.dev_status = a->dev_status;
  j.q_pos = a->q_pos;
  return j;
}

static hyb::AttendJob swa_job(const hyb_swa_args* a) {
  hyb::AttendJob j{};
  j.mode = 2, j.q = a->q, j.k = a->kw, j.v = a->vw, j.o_in = a->o_in, j.lse_in = a->lse_in, j.out = a->out;
  j.out_bf16 = a->out_dtype == HYB_BF16, j.lse = a->lse_out;
  j.batch = a->batch, j.n_q = a->n_q, j.n_h = a->n_h, j.c = a->c, j.n_entries = a->n_kv, j.kv_stride = a->n_kv;
  j.kv_pos0 = a->kv_pos0, j.q_pos0 = a->q_pos0, j.n_win = a->n_win;
  j.scale = a->scale, j.dtype = a->dtype, j.dev_status = a->dev_status;
  j.q_pos = a->q_pos, j.kv_pos0s = a->kv_pos0s;
  return j;
}

static hyb_status validate_attend_common(const char* name, int64_t batch, int64_t n_q, int64_t n_h, int64_t c,
                                         int32_t dtype, const void* q, const void* k, const void* v) {
  if (batch < 0 || n_q < 0 || n_h < 0 || c < 1) return fail(HYB_ERR_INVALID_ARG, "%s: negative size or c < 1", name);
  if (dtype != HYB_F32 && dtype != HYB_BF16) return fail(HYB_ERR_INVALID_ARG, "%s: dtype must be F32 or BF16", name);
  if (!hyb::attend_cc_shape_supported(c, n_h))
    return fail(HYB_ERR_UNSUPPORTED, "%s: c = %lld not compiled (32, 64, 128, 256, 512)", name, (long long)c);
  if (batch == 0 || n_q == 0 || n_h == 0) return ok();
  if (!q || !k || !v) return fail(HYB_ERR_INVALID_ARG, "%s: NULL q/k/v", name);
  const size_t al = lane_align(c, dtype);
  if (!aligned(q, al) || !aligned(k, al) || !aligned(v, al)) return fail(HYB_ERR_INVALID_ARG, "%s: misaligned q/k/v", name);
  return ok();
}

// Attention dispatch: the tensor-core kernel for its shapes (bf16, c = 512,
// heads a multiple of 64), the CUDA-core kernel otherwise.  The workspace of
// csa_attend / hca_attend starts with the tensor-core kernel's join counters
// (kJoinRegionBytes, zero between calls) whichever kernel runs; other scratch
// follows them.  A standalone window merge has no join.
static size_t join_region(const hyb::AttendJob& j) { return j.mode == 2 ? 0 : hyb::kJoinRegionBytes; }

// The 128-head kernel serves its shapes when it is enabled (HYB_ATTEND_H128, on by default).
static bool use_h128(const hyb::AttendJob& j) { return hyb::attend_h128_enabled() && hyb::attend_h128_supported(j); }

static size_t attend_workspace(const hyb::AttendJob& j) {
  if (use_h128(j)) return hyb::attend_h128_workspace_bytes(j);
  return hyb::attend_tc_supported(j) ? hyb::attend_tc_workspace_bytes(j)
                                     : join_region(j) + hyb::attend_cc_workspace_bytes(j);
}

static cudaError_t launch_attend(const hyb::AttendJob& j, void* ws, cudaStream_t s) {
  if (use_h128(j)) return hyb::launch_attend_h128(j, ws, s);
  if (hyb::attend_tc_supported(j)) return hyb::launch_attend_tc(j, ws, s);
  return hyb::launch_attend_cc(j, static_cast<char*>(ws) + join_region(j), s);
}

// sink / sink_done: a per-head sink that the launched kernel joins to its final result
// where it can (the 128-head kernel); *sink_done says whether it did.
static hyb_status run_attend(const char* name, hyb::AttendJob j, void* workspace, size_t ws_bytes, void* stream,
                             const float* sink = nullptr, bool* sink_done = nullptr) {
  const size_t need = attend_workspace(j);
  if (need > 0 && (!workspace || ws_bytes < need))
    return fail(HYB_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
  if (!aligned(workspace, 256)) return fail(HYB_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", name);
  if (sink && use_h128(j)) {
    j.sink = sink;
    *sink_done = true;
  }
  return cuda_status(launch_attend(j, workspace, static_cast<cudaStream_t>(stream)), name);
}

// ------------------------------------------------- fused window merge

static hyb::AttendJob fused_job(hyb::AttendJob j, const hyb_window* w) {
  j.win = 1, j.wk = w->kw, j.w_stride = w->n_kv, j.w_pos0 = w->kv_pos0, j.wq_pos0 = w->q_pos0, j.n_win = w->n_win;
  j.wq_pos = w->q_pos, j.w_pos0s = w->kv_pos0s;
  j.out = w->out, j.out_bf16 = w->out_dtype == HYB_BF16, j.o = nullptr;
  return j;
}

// the two-step fallback's window merge over the compressed result (o_in, lse_in)
static hyb::AttendJob window_merge_job(const hyb::AttendJob& c, const hyb_window* w, const float* o_in,
                                       const float* lse_in, float* lse_out) {
  hyb::AttendJob j{};
  j.mode = 2, j.q = c.q, j.k = w->kw, j.v = w->kw, j.o_in = o_in, j.lse_in = lse_in, j.out = w->out;
  j.out_bf16 = w->out_dtype == HYB_BF16, j.lse = lse_out;
  j.batch = c.batch, j.n_q = c.n_q, j.n_h = c.n_h, j.c = c.c, j.n_entries = w->n_kv, j.kv_stride = w->n_kv;
  j.kv_pos0 = w->kv_pos0, j.q_pos0 = w->q_pos0, j.n_win = w->n_win;
  j.scale = c.scale, j.dtype = c.dtype, j.dev_status = c.dev_status;
  j.q_pos = w->q_pos, j.kv_pos0s = w->kv_pos0s;
  return j;
}

static size_t fallback_io_bytes(const hyb::AttendJob& c) {
  const size_t n = (size_t)(c.batch * c.n_q * c.n_h);
  return round_up(n * (size_t)c.c * sizeof(float), 256) + round_up(n * sizeof(float), 256);
}

static size_t attend_window_workspace(const hyb::AttendJob& c, const hyb_window* w) {
  const hyb::AttendJob f = fused_job(c, w);
  if (use_h128(f)) return hyb::attend_h128_workspace_bytes(f);
  if (hyb::attend_tc_supported(f)) return hyb::attend_tc_workspace_bytes(f);
  const hyb::AttendJob m = window_merge_job(c, w, nullptr, nullptr, nullptr);
  return round_up(std::max(attend_workspace(c), hyb::kJoinRegionBytes + attend_workspace(m)), 256) +
         fallback_io_bytes(c);
}

static hyb_status validate_window(const char* name, const hyb::AttendJob& c, const hyb_window* w) {
  if (w->n_win < 1 || w->q_pos0 < 0 || w->kv_pos0 < 0 || w->n_kv < 0)
    return fail(HYB_ERR_INVALID_ARG, "%s: window n_win < 1 or negative position", name);
  if (w->out_dtype != HYB_F32 && w->out_dtype != HYB_BF16)
    return fail(HYB_ERR_INVALID_ARG, "%s: window out_dtype must be F32 or BF16", name);
  if (c.mode == 1 && (w->q_pos != c.q_pos || (!c.q_pos && w->q_pos0 != c.q_pos0)))
    return fail(HYB_ERR_INVALID_ARG, "%s: the window's query positions (q_pos0 %lld, q_pos %p) differ from the call's "
                "(q_pos0 %lld, q_pos %p)", name, (long long)w->q_pos0, (const void*)w->q_pos, (long long)c.q_pos0,
                (const void*)c.q_pos);
  if (!aligned(w->q_pos, 8) || !aligned(w->kv_pos0s, 8))
    return fail(HYB_ERR_INVALID_ARG, "%s: misaligned window q_pos/kv_pos0s", name);
  if (c.batch == 0 || c.n_q == 0 || c.n_h == 0) return ok();
  const int64_t lo = w->q_pos0 - w->n_win + 1 > 0 ? w->q_pos0 - w->n_win + 1 : 0;
  const int64_t hi = w->q_pos0 + c.n_q - 1;
  // (positions in device memory are checked by the kernels)
  if (!w->q_pos && !w->kv_pos0s && (lo < w->kv_pos0 || hi >= w->kv_pos0 + w->n_kv))
    return fail(HYB_ERR_INVALID_ARG, "%s: window rows %lld..%lld are not all inside the buffer %lld..%lld", name,
                (long long)lo, (long long)hi, (long long)w->kv_pos0, (long long)(w->kv_pos0 + w->n_kv - 1));
  if (!w->kw || !w->out) return fail(HYB_ERR_INVALID_ARG, "%s: NULL window kw/out", name);
  if (!aligned(w->kw, lane_align(c.c, c.dtype)) || !aligned(w->out, lane_align(c.c, w->out_dtype)))
    return fail(HYB_ERR_INVALID_ARG, "%s: misaligned window kw/out", name);
  return ok();
}

// c: the compressed-branch job (its o unused), lse: the union's lse
static hyb_status run_attend_window(const char* name, hyb::AttendJob c, const hyb_window* w, void* workspace,
                                    size_t ws_bytes, void* stream, const float* sink = nullptr,
                                    bool* sink_done = nullptr) {
  const size_t need = attend_window_workspace(c, w);
  if (need > 0 && (!workspace || ws_bytes < need))
    return fail(HYB_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
  if (!aligned(workspace, 256)) return fail(HYB_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  hyb::AttendJob f = fused_job(c, w);
  if (use_h128(f)) {
    if (sink) f.sink = sink, *sink_done = true;
    return cuda_status(hyb::launch_attend_h128(f, workspace, s), name);
  }
  if (hyb::attend_tc_supported(f)) return cuda_status(hyb::launch_attend_tc(f, workspace, s), name);
  // two steps: the compressed branch into the workspace (after the kernels' own
  // scratch, which keeps the join counters first), then the window merge
  const size_t n = (size_t)(c.batch * c.n_q * c.n_h);
  const hyb::AttendJob m0 = window_merge_job(c, w, nullptr, nullptr, nullptr);
  char* base = static_cast<char*>(workspace);
  char* io = base + round_up(std::max(attend_workspace(c), hyb::kJoinRegionBytes + attend_workspace(m0)), 256);
  float* o_tmp = reinterpret_cast<float*>(io);
  float* lse_tmp = reinterpret_cast<float*>(io + round_up(n * (size_t)c.c * sizeof(float), 256));
  float* lse_out = c.lse;
  c.o = o_tmp, c.lse = lse_tmp;
  cudaError_t e = launch_attend(c, base, s);
  if (e != cudaSuccess) return cuda_status(e, name);
  const hyb::AttendJob m = window_merge_job(c, w, o_tmp, lse_tmp, lse_out);
  return cuda_status(launch_attend(m, base + hyb::kJoinRegionBytes, s), name);  // (the counters stay untouched)
}

size_t csa_attend_workspace_size(const hyb_csa_attend_args* a) {
  if (!a || a->batch <= 0 || a->n_q <= 0 || a->n_h <= 0) return 0;
  if (a->window) return attend_window_workspace(csa_job(a), a->window);
  return attend_workspace(csa_job(a));
}

// The attention sink on a call's final result: the fused window's out where there is
// one, else o (float32), and lse.
static hyb_status apply_sink(const char* name, const hyb_window* w, float* o, float* lse, const float* sink,
                             int64_t rows, int64_t n_h, int64_t c, void* stream) {
  void* out = w ? w->out : static_cast<void*>(o);
  const int32_t dt = w ? w->out_dtype : HYB_F32;
  return cuda_status(hyb::launch_sink(out, dt, lse, sink, rows * n_h, n_h, c, static_cast<cudaStream_t>(stream)), name);
}

hyb_status csa_attend(const hyb_csa_attend_args* a, void* workspace, size_t ws_bytes, void* stream) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "csa_attend: args is NULL");
  hyb_status st = validate_attend_common("csa_attend", a->batch, a->n_q, a->n_h, a->c, a->dtype, a->q, a->kc, a->vc);
  if (st != HYB_OK) return st;
  if (a->k < 0 || a->n_entries < 0 || a->kv_stride < 0) return fail(HYB_ERR_INVALID_ARG, "csa_attend: negative size");
  if (a->kv_stride != 0 && a->kv_stride < a->n_entries) return fail(HYB_ERR_INVALID_ARG, "csa_attend: kv_stride < n_entries");
  if (a->window && (st = validate_window("csa_attend", csa_job(a), a->window)) != HYB_OK) return st;
  if (a->batch == 0 || a->n_q == 0 || a->n_h == 0) return ok();
  if ((!a->o && !a->window) || !a->lse || (a->k > 0 && !a->idx))
    return fail(HYB_ERR_INVALID_ARG, "csa_attend: NULL o/lse/idx");
  if (!aligned(a->o, lane_align(a->c, HYB_F32)) || !aligned(a->idx, 4) || !aligned(a->lse, 4) || !aligned(a->sink, 4))
    return fail(HYB_ERR_INVALID_ARG, "csa_attend: misaligned o/lse/idx/sink");
  bool sink_done = false;
  st = a->window ? run_attend_window("csa_attend", csa_job(a), a->window, workspace, ws_bytes, stream, a->sink, &sink_done)
                 : run_attend("csa_attend", csa_job(a), workspace, ws_bytes, stream, a->sink, &sink_done);
  if (st != HYB_OK || !a->sink || sink_done) return st;
  return apply_sink("csa_attend", a->window, a->o, a->lse, a->sink, a->batch * a->n_q, a->n_h, a->c, stream);
}

size_t hca_attend_workspace_size(const hyb_hca_attend_args* a) {
  if (!a || a->batch <= 0 || a->n_q <= 0 || a->n_h <= 0 || a->m < 1) return 0;
  if (a->window) return attend_window_workspace(hca_job(a), a->window);
  return attend_workspace(hca_job(a));
}

hyb_status hca_attend(const hyb_hca_attend_args* a, void* workspace, size_t ws_bytes, void* stream) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "hca_attend: args is NULL");
  hyb_status st = validate_attend_common("hca_attend", a->batch, a->n_q, a->n_h, a->c, a->dtype, a->q, a->kc, a->vc);
  if (st != HYB_OK) return st;
  if (a->m < 1 || a->q_pos0 < 0 || a->n_entries < 0 || a->kv_stride < 0)
    return fail(HYB_ERR_INVALID_ARG, "hca_attend: m < 1 or negative size");
  if (a->kv_stride != 0 && a->kv_stride < a->n_entries) return fail(HYB_ERR_INVALID_ARG, "hca_attend: kv_stride < n_entries");
  if (!aligned(a->q_pos, 8)) return fail(HYB_ERR_INVALID_ARG, "hca_attend: misaligned q_pos");
  if (!a->q_pos && a->n_q > 0 && hyb::visible_entries(a->q_pos0 + a->n_q - 1, a->m) > a->n_entries)
    return fail(HYB_ERR_INVALID_ARG, "hca_attend: the last query sees %lld entries but only %lld exist",
                (long long)hyb::visible_entries(a->q_pos0 + a->n_q - 1, a->m), (long long)a->n_entries);
  if (a->window && (st = validate_window("hca_attend", hca_job(a), a->window)) != HYB_OK) return st;
  if (a->batch == 0 || a->n_q == 0 || a->n_h == 0) return ok();
  if ((!a->o && !a->window) || !a->lse) return fail(HYB_ERR_INVALID_ARG, "hca_attend: NULL o/lse");
  if (!aligned(a->o, lane_align(a->c, HYB_F32)) || !aligned(a->lse, 4) || !aligned(a->sink, 4))
    return fail(HYB_ERR_INVALID_ARG, "hca_attend: misaligned o/lse/sink");
  bool sink_done = false;
  st = a->window ? run_attend_window("hca_attend", hca_job(a), a->window, workspace, ws_bytes, stream, a->sink, &sink_done)
                 : run_attend("hca_attend", hca_job(a), workspace, ws_bytes, stream, a->sink, &sink_done);
  if (st != HYB_OK || !a->sink || sink_done) return st;
  return apply_sink("hca_attend", a->window, a->o, a->lse, a->sink, a->batch * a->n_q, a->n_h, a->c, stream);
}

size_t swa_merge_workspace_size(const hyb_swa_args* a) {
  if (!a || a->batch <= 0 || a->n_q <= 0 || a->n_h <= 0) return 0;
  return attend_workspace(swa_job(a));
}

hyb_status swa_merge(const hyb_swa_args* a, void* workspace, size_t ws_bytes, void* stream) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "swa_merge: args is NULL");
  hyb_status st = validate_attend_common("swa_merge", a->batch, a->n_q, a->n_h, a->c, a->dtype, a->q, a->kw, a->vw);
  if (st != HYB_OK) return st;
  if (a->n_win < 1 || a->q_pos0 < 0 || a->kv_pos0 < 0 || a->n_kv < 0)
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: n_win < 1 or negative position");
  if (a->out_dtype != HYB_F32 && a->out_dtype != HYB_BF16)
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: out_dtype must be F32 or BF16");
  if ((a->o_in == nullptr) != (a->lse_in == nullptr))
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: o_in and lse_in must both be given or both be NULL");
  if (a->batch == 0 || a->n_q == 0 || a->n_h == 0) return ok();
  if (!aligned(a->q_pos, 8) || !aligned(a->kv_pos0s, 8))
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: misaligned q_pos/kv_pos0s");
  const int64_t lo = a->q_pos0 - a->n_win + 1 > 0 ? a->q_pos0 - a->n_win + 1 : 0;
  const int64_t hi = a->q_pos0 + a->n_q - 1;
  // (positions in device memory are checked by the kernels)
  if (!a->q_pos && !a->kv_pos0s && (lo < a->kv_pos0 || hi >= a->kv_pos0 + a->n_kv))
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: window rows %lld..%lld are not all inside the buffer %lld..%lld",
                (long long)lo, (long long)hi, (long long)a->kv_pos0, (long long)(a->kv_pos0 + a->n_kv - 1));
  if (!a->out) return fail(HYB_ERR_INVALID_ARG, "swa_merge: NULL out");
  if (!aligned(a->out, lane_align(a->c, a->out_dtype)) || !aligned(a->o_in, lane_align(a->c, HYB_F32)) ||
      !aligned(a->lse_in, 4) || !aligned(a->lse_out, 4))
    return fail(HYB_ERR_INVALID_ARG, "swa_merge: misaligned out/o_in/lse");
  return run_attend("swa_merge", swa_job(a), workspace, ws_bytes, stream);
}

// ------------------------------------------------- grouped output projection

hyb_status hyb_grouped_out_proj(const hyb_gproj_args* a, void* stream) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: args is NULL");
  if (a->rows < 0 || a->n_h < 1 || a->c < 1 || a->g < 1 || a->d_g < 1 || a->out_row_stride < 0)
    return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: negative size or n_h, c, g, d_g < 1");
  if (a->n_h % a->g != 0) return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: g must divide n_h");
  if (a->dtype != HYB_BF16) return fail(HYB_ERR_UNSUPPORTED, "hyb_grouped_out_proj: o and w must be BF16");
  if (a->out_dtype != HYB_F32 && a->out_dtype != HYB_BF16)
    return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: out_dtype must be F32 or BF16");
  if (!hyb::out_proj_shape_supported(a->n_h, a->c, a->g, a->d_g))
    return fail(HYB_ERR_UNSUPPORTED, "hyb_grouped_out_proj: d_g = %lld (a multiple of 128 needed) / group inputs %lld "
                "(a multiple of 64 needed)", (long long)a->d_g, (long long)(a->n_h / a->g * a->c));
  if (a->rows == 0) return ok();
  if (!a->o || !a->w || !a->out) return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: NULL o/w/out");
  if (!aligned(a->o, 16) || !aligned(a->w, 16) || !aligned(a->out, 16))
    return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: pointers must be 16-byte aligned");
  if (a->rows >= (int64_t(1) << 31) || a->g * a->d_g >= (int64_t(1) << 31))
    return fail(HYB_ERR_UNSUPPORTED, "hyb_grouped_out_proj: too many rows or features");
  if (a->out_row_stride != 0 && a->out_row_stride < a->g * a->d_g)
    return fail(HYB_ERR_INVALID_ARG, "hyb_grouped_out_proj: out_row_stride %lld < g*d_g = %lld",
                (long long)a->out_row_stride, (long long)(a->g * a->d_g));
  const int64_t stride = a->out_row_stride ? a->out_row_stride : a->g * a->d_g;
  return cuda_status(hyb::launch_out_proj(a->o, a->w, a->out, a->out_dtype == HYB_BF16, a->rows, a->n_h, a->c, a->g,
                                          a->d_g, stride, a->dev_status, static_cast<cudaStream_t>(stream)),
                     "hyb_grouped_out_proj");
}

// ---------------------------------------------------------- RMSNorm + RoPE

static hyb_status check_norm_rope(const hyb_norm_rope_args* a) {
  if (!a) return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: args is NULL");
  if (a->rows < 0 || a->c < 2 || a->c % 2 != 0)
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: rows < 0 or c not even and >= 2");
  if (a->dtype != HYB_F32 && a->dtype != HYB_BF16)
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: dtype must be F32 or BF16");
  if (!(a->eps >= 0.f) || !std::isfinite(a->eps)) return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: eps must be >= 0");
  if (a->rope_dims < 0 || a->rope_dims % 2 != 0 || a->rope_dims > a->c)
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: rope_dims must be even and <= c");
  if (a->rope_dims > 0 && (!a->pos || a->rows_per_pos < 1 || !(a->theta > 0.0)))
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: rotation needs pos, rows_per_pos >= 1 and theta > 0");
  if (a->row_stride != 0 && (a->row_stride < a->c || a->row_stride % 2 != 0))
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: row_stride must be 0 or an even number >= c");
  if (a->rows == 0) return ok();
  if (!a->x) return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: x is NULL");
  if (!aligned(a->x, 2 * elem_size(a->dtype)) || !aligned(a->gamma, 4) || !aligned(a->pos, 8))
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope: misaligned x/gamma/pos");
  return ok();
}

hyb_status hyb_rmsnorm_rope(const hyb_norm_rope_args* a, void* stream) {
  const hyb_status st = check_norm_rope(a);
  if (st != HYB_OK || a->rows == 0) return st;
  return cuda_status(hyb::launch_norm_rope(a, static_cast<cudaStream_t>(stream)), "hyb_rmsnorm_rope");
}

hyb_status hyb_rmsnorm_rope_batch(const hyb_norm_rope_args* calls, int32_t n_calls, void* stream) {
  static_assert(HYB_NORM_ROPE_BATCH_MAX == hyb::kNormRopeBatchMax, "batch size");
  if (n_calls < 0 || n_calls > HYB_NORM_ROPE_BATCH_MAX)
    return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope_batch: n_calls must be 0 .. HYB_NORM_ROPE_BATCH_MAX");
  if (n_calls == 0) return ok();
  if (!calls) return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope_batch: calls is NULL");
  for (int32_t i = 0; i < n_calls; ++i) {
    const hyb_status st = check_norm_rope(&calls[i]);
    if (st != HYB_OK) return st;
    if (calls[i].dtype != calls[0].dtype)
      return fail(HYB_ERR_INVALID_ARG, "hyb_rmsnorm_rope_batch: the calls must share one dtype");
  }
  return cuda_status(hyb::launch_norm_rope_batch(calls, n_calls, static_cast<cudaStream_t>(stream)),
                     "hyb_rmsnorm_rope_batch");
}

}  // extern "C"
