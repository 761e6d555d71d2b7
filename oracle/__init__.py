"""Float64 CPU oracle for the DeepSeek-V4 hybrid-attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never calls it and
it never calls the CUDA library: the two share no code.

The arithmetic lives in ``hyb_oracle.c`` (plain C, float64, one thread); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  Every function names the page section it restates; see the header of
``hyb_oracle.c`` for the readings taken where the pages are silent.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(page-printed worked examples, closed forms, reductions to library routines,
brute force); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hyb_oracle.c")
_LIB = os.path.join(_HERE, "libhyb_oracle.so")

F32, BF16, E4M3 = 0, 1, 2  # the oracle's own dtype codes

_lock = threading.Lock()
_lib = None

_GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no contraction)."""
    cmd = ["gcc", *_GCC_FLAGS, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def load(path: str | None = None):
    """Load (building if missing or stale) the oracle shared library."""
    global _lib
    if path is None:
        path = os.environ.get("HYB_ORACLE_LIB")  # lets a test load a deliberately broken copy
    if path is not None:
        with _lock:
            if _lib is None:
                _lib = _declare(ctypes.CDLL(path))
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i = ctypes.c_int
_d = ctypes.c_double


def _declare(lib):
    lib.orc_bf16_decode.restype = _d
    lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.orc_e4m3_decode.restype = _d
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_round_bf16.restype = _d
    lib.orc_round_bf16.argtypes = [_d]
    lib.orc_compress_out_count.restype = _i64
    lib.orc_compress_out_count.argtypes = [_i64, _i64, _i, _i64]
    lib.orc_visible.restype = _i64
    lib.orc_visible.argtypes = [_i64, _i64]
    lib.orc_window_count.restype = _i64
    lib.orc_window_count.argtypes = [_i64, _i64]
    lib.orc_compress.restype = None
    lib.orc_compress.argtypes = [_i, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i, _i64, _p]
    lib.orc_compress_weights.restype = None
    lib.orc_compress_weights.argtypes = [_i, _p, _p, _p, _i64, _i64, _i64, _i, _i64, _i64, _i64, _i64, _p]
    lib.orc_quantise_fp8_rows.restype = None
    lib.orc_quantise_fp8_rows.argtypes = [_p, _i64, _i64, _p, _p]
    lib.orc_index_scores.restype = None
    lib.orc_index_scores.argtypes = [_i, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]
    lib.orc_topk.restype = None
    lib.orc_topk.argtypes = [_p, _p, _i64, _i64, _i64, _p]
    lib.orc_csa_attend.restype = None
    lib.orc_csa_attend.argtypes = [_i, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _d, _p, _p]
    lib.orc_hca_attend.restype = None
    lib.orc_hca_attend.argtypes = [_i, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _d, _p, _p]
    lib.orc_swa_merge.restype = None
    lib.orc_swa_merge.argtypes = [_i, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _d, _p, _p,
                                  _p, _p]
    lib.orc_rmsnorm.restype = None
    lib.orc_rmsnorm.argtypes = [_p, _i64, _i64, _p, _d, _p]
    lib.orc_rope_partial.restype = None
    lib.orc_rope_partial.argtypes = [_p, _i64, _i64, _i64, _p, _d, _p]
    lib.orc_sink_merge.restype = None
    lib.orc_sink_merge.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _p]
    lib.orc_e2m1_decode.restype = _d
    lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e8m0_decode.restype = _d
    lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
    lib.orc_quantise_mxfp4_rows.restype = None
    lib.orc_quantise_mxfp4_rows.argtypes = [_p, _i64, _i64, _p, _p]
    lib.orc_grouped_out_proj.restype = None
    lib.orc_grouped_out_proj.argtypes = [_p, _p, _i64, _i64, _i64, _i64, _i64, _p]
    return lib


# ----------------------------------------------------------------- helpers

_NP_OF = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8}


def _arr(x, dtype_code=None, np_dtype=None):
    """Contiguous numpy view of x holding the raw element bits the oracle decodes."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (CPU) -> raw bits
        import torch

        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            x = t.view(torch.int16).numpy().view(np.uint16)
        elif t.dtype == torch.float8_e4m3fn:
            x = t.view(torch.uint8).numpy()
        else:
            x = t.numpy()
    want = np_dtype if np_dtype is not None else _NP_OF[dtype_code]
    a = np.ascontiguousarray(x)
    if a.dtype != want:
        if want in (np.uint16, np.uint8) and a.dtype.itemsize == np.dtype(want).itemsize:
            a = a.view(want)
        else:
            a = a.astype(want)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def dtype_code(x) -> int:
    """Oracle dtype code for a torch tensor or numpy array holding raw values."""
    if hasattr(x, "dtype") and hasattr(x, "detach"):
        import torch

        return {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}[x.dtype]
    return {np.dtype(np.float32): F32, np.dtype(np.uint16): BF16, np.dtype(np.uint8): E4M3}[np.dtype(x.dtype)]


# --------------------------------------------------------------- formats


def bf16_decode(bits) -> np.ndarray:
    lib = load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.orc_bf16_decode(int(v)) for v in b]).reshape(np.shape(bits))


def e4m3_decode(codes) -> np.ndarray:
    lib = load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c]).reshape(np.shape(codes))


def e4m3_encode(x) -> np.ndarray:
    lib = load()
    v = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_e4m3_encode(float(e)) for e in v], dtype=np.uint8).reshape(np.shape(x))


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even)."""
    lib = load()
    v = np.asarray(x, dtype=np.float64)
    flat = v.ravel()
    return np.array([lib.orc_round_bf16(float(e)) for e in flat]).reshape(v.shape)


def round_bf16_bits(x) -> np.ndarray:
    """The bf16 bit patterns (uint16) of round_bf16(x)."""
    r = round_bf16(x).astype(np.float32)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# -------------------------------------------------------------- counting


def compress_out_count(n_rows: int, m: int, overlap: bool, first_block: int = 0) -> int:
    return int(load().orc_compress_out_count(n_rows, m, int(bool(overlap)), first_block))


def visible(t: int, m: int) -> int:
    return int(load().orc_visible(t, m))


def window_count(t: int, n_win: int) -> int:
    return int(load().orc_window_count(t, n_win))


# -------------------------------------------------------------- compress


def compress(ca, za, bias, m: int, cb=None, zb=None, overlap: bool = False, first_block: int = 0) -> np.ndarray:
    """Softmax-gated compressor (pages: trishampatil.com section V.1 / VI).

    ca, za (and cb, zb when overlap) are [B][n][c] float32 / bf16-bits arrays;
    bias is [2m or m][c] float32.  Returns [B][n_out][c] float64."""
    code = dtype_code(ca)
    ca_, za_ = _arr(ca, code), _arr(za, code)
    cb_ = _arr(cb, code) if overlap else None
    zb_ = _arr(zb, code) if overlap else None
    bias_ = _arr(bias, np_dtype=np.float32)
    B, n, c = ca_.shape
    n_out = compress_out_count(n, m, overlap, first_block)
    out = np.zeros((B, n_out, c), dtype=np.float64)
    load().orc_compress(code, _ptr(ca_), _ptr(cb_), _ptr(za_), _ptr(zb_), _ptr(bias_), B, n, c, m, int(bool(overlap)),
                        first_block, _ptr(out))
    return out


def compress_weights(za, bias, m: int, b: int, j: int, ch: int, zb=None, overlap: bool = False,
                     first_block: int = 0) -> np.ndarray:
    code = dtype_code(za)
    za_ = _arr(za, code)
    zb_ = _arr(zb, code) if overlap else None
    bias_ = _arr(bias, np_dtype=np.float32)
    _, n, c = za_.shape
    w = np.zeros(2 * m if overlap else m)
    load().orc_compress_weights(code, _ptr(za_), _ptr(zb_), _ptr(bias_), n, c, m, int(bool(overlap)), first_block, b,
                                j, ch, _ptr(w))
    return w


def quantise_fp8_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Row-wise e4m3 quantiser; decisions in float32 (see hyb_oracle.c, R9)."""
    x_ = np.ascontiguousarray(x, dtype=np.float32)
    shp = x_.shape
    rows = int(np.prod(shp[:-1]))
    c = shp[-1]
    codes = np.zeros(shp, dtype=np.uint8)
    scales = np.zeros(shp[:-1], dtype=np.float32)
    load().orc_quantise_fp8_rows(_ptr(x_), rows, c, _ptr(codes), _ptr(scales))
    return codes, scales


# ------------------------------------------------------------------ index


def index_scores(qI, w, kI, m: int, q_pos0: int, qI_scale=None, kI_scale=None) -> np.ndarray:
    """Lightning-indexer scores (trishampatil.com section V.2); -inf where not visible.

    qI [B][n_q][n_ih][c_I], kI [B][N][c_I] as float32 or e4m3 codes (uint8 /
    torch float8); w [B][n_q][n_ih] float32.  Returns [B][n_q][N] float64."""
    code = dtype_code(qI)
    qI_, kI_ = _arr(qI, code), _arr(kI, code)
    w_ = _arr(w, np_dtype=np.float32)
    qs = _arr(qI_scale, np_dtype=np.float32) if code == E4M3 else None
    ks = _arr(kI_scale, np_dtype=np.float32) if code == E4M3 else None
    B, n_q, n_ih, c_I = qI_.shape
    N = kI_.shape[1]
    out = np.zeros((B, n_q, N), dtype=np.float64)
    load().orc_index_scores(code, _ptr(qI_), _ptr(qs), _ptr(w_), _ptr(kI_), _ptr(ks), B, n_q, N, n_ih, c_I, m,
                            q_pos0, _ptr(out))
    return out


def topk(scores, visible_counts, k: int) -> np.ndarray:
    """Top-k selector (reading R6 in hyb_oracle.c).  scores [..., N] float64;
    visible_counts broadcastable to scores.shape[:-1].  Returns int32 [..., k]."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    lead = s.shape[:-1]
    N = s.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    vis = np.ascontiguousarray(np.broadcast_to(np.asarray(visible_counts, dtype=np.int64), lead)).reshape(-1)
    idx = np.zeros((rows, k), dtype=np.int32)
    load().orc_topk(_ptr(s), _ptr(vis), rows, N, k, _ptr(idx))
    return idx.reshape(*lead, k)


# -------------------------------------------------------------- attention


def csa_attend(q, kc, vc, idx, scale: float):
    """CSA core attention over selected entries (trishampatil.com section V.3)."""
    code = dtype_code(q)
    q_, k_, v_ = _arr(q, code), _arr(kc, code), _arr(vc, code)
    idx_ = _arr(idx, np_dtype=np.int32)
    B, n_q, n_h, c = q_.shape
    N = k_.shape[1]
    k = idx_.shape[-1]
    o = np.zeros((B, n_q, n_h, c))
    lse = np.zeros((B, n_q, n_h))
    load().orc_csa_attend(code, _ptr(q_), _ptr(k_), _ptr(v_), _ptr(idx_), B, n_q, n_h, c, N, k, float(scale), _ptr(o),
                          _ptr(lse))
    return o, lse


def hca_attend(q, kc, vc, m: int, q_pos0: int, scale: float):
    """HCA core attention over all visible entries (trishampatil.com section VI)."""
    code = dtype_code(q)
    q_, k_, v_ = _arr(q, code), _arr(kc, code), _arr(vc, code)
    B, n_q, n_h, c = q_.shape
    N = k_.shape[1]
    o = np.zeros((B, n_q, n_h, c))
    lse = np.zeros((B, n_q, n_h))
    load().orc_hca_attend(code, _ptr(q_), _ptr(k_), _ptr(v_), B, n_q, n_h, c, N, m, q_pos0, float(scale), _ptr(o),
                          _ptr(lse))
    return o, lse


def swa_merge(q, kw, vw, kv_pos0: int, q_pos0: int, n_win: int, scale: float, o_in, lse_in):
    """Sliding-window branch merged by log-sum-exp (modernaiengineering.com,
    "One query in a CSA layer", steps 4-5).  Returns (out, lse) float64."""
    code = dtype_code(q)
    q_, kw_, vw_ = _arr(q, code), _arr(kw, code), _arr(vw, code)
    B, n_q, n_h, c = q_.shape
    n_kv = kw_.shape[1]
    o_in_ = np.ascontiguousarray(o_in, dtype=np.float64)
    lse_in_ = np.ascontiguousarray(lse_in, dtype=np.float64)
    out = np.zeros((B, n_q, n_h, c))
    lse = np.zeros((B, n_q, n_h))
    load().orc_swa_merge(code, _ptr(q_), _ptr(kw_), _ptr(vw_), B, n_q, n_h, c, n_kv, kv_pos0, q_pos0, n_win,
                         float(scale), _ptr(o_in_), _ptr(lse_in_), _ptr(out), _ptr(lse))
    return out, lse


# ------------------------------------------------------ in-branch operations


def rmsnorm(x, gamma=None, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm over the last dimension ("DeepSeek-V4 hybrid attention" (trishampatil.com)
    section IV: queries and compressed KV entries are RMS-normalised inside both branches).
    Returns float64 of x's shape."""
    x_ = np.ascontiguousarray(x, dtype=np.float64)
    c = x_.shape[-1]
    rows = int(np.prod(x_.shape[:-1])) if x_.ndim > 1 else 1
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64)
    y = np.zeros_like(x_)
    load().orc_rmsnorm(_ptr(x_), rows, c, _ptr(g), float(eps), _ptr(y))
    return y


def rope_partial(x, pos, rope_dims: int = 64, theta: float = 10000.0) -> np.ndarray:
    """Rotary encoding of the last rope_dims dimensions only (same page, section IV:
    "partial RoPE"), consecutive pairs rotated by pos * theta^(-2i/rope_dims) (the
    pairing and frequencies of the PyTorch walkthrough on juhe.plus, "The Code: RoPE
    Helpers").  x [..., c]; pos broadcastable to x.shape[:-1].  Returns float64."""
    x_ = np.ascontiguousarray(x, dtype=np.float64)
    c = x_.shape[-1]
    lead = x_.shape[:-1]
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.float64), lead)).reshape(-1)
    y = np.zeros_like(x_)
    load().orc_rope_partial(_ptr(x_), int(p.size), c, rope_dims, _ptr(p), float(theta), _ptr(y))
    return y


def sink_merge(o, lse, sink):
    """Per-head attention sink (same page, section IV): one more logit per head in the
    softmax denominator with no value.  o [..., n_h, c], lse [..., n_h], sink [n_h].
    Returns (out, lse) float64."""
    o_ = np.ascontiguousarray(o, dtype=np.float64)
    l_ = np.ascontiguousarray(lse, dtype=np.float64)
    s_ = np.ascontiguousarray(sink, dtype=np.float64)
    n_h, c = o_.shape[-2], o_.shape[-1]
    rows = int(np.prod(o_.shape[:-2])) if o_.ndim > 2 else 1
    out = np.zeros_like(o_)
    lo = np.zeros_like(l_)
    load().orc_sink_merge(_ptr(o_), _ptr(l_), rows, n_h, c, _ptr(s_), _ptr(out), _ptr(lo))
    return out, lo


def grouped_out_proj(o, W, W_out=None) -> np.ndarray:
    """Grouped output projection ("DeepSeek-V4 hybrid attention" (trishampatil.com)
    section V.3): o [..., n_h, c] (the heads of each row), W [g, d_g, (n_h/g)*c]: group j
    of n_h/g consecutive heads projected by W[j]; the g results concatenated
    ([..., g*d_g]), then, when W_out [d, g*d_g] is given, mapped to d by that matrix (a
    library matmul).  Returns float64."""
    o_ = np.ascontiguousarray(o, dtype=np.float64)
    W_ = np.ascontiguousarray(W, dtype=np.float64)
    n_h, c = o_.shape[-2], o_.shape[-1]
    g, d_g, in_g = W_.shape
    if n_h % g or in_g != (n_h // g) * c:
        raise ValueError("W must be [g, d_g, (n_h/g)*c] with g dividing n_h")
    lead = o_.shape[:-2]
    rows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (g * d_g,))
    load().orc_grouped_out_proj(_ptr(o_), _ptr(W_), rows, n_h, c, g, d_g, _ptr(out))
    if W_out is not None:
        out = out @ np.asarray(W_out, dtype=np.float64).T
    return out


# ------------------------------------------------------------------ MXFP4


def e2m1_decode(codes) -> np.ndarray:
    """Values of e2m1 codes (one per byte), each decoded by the C decoder (a table of its 16
    results, indexed by code)."""
    lib = load()
    table = np.array([lib.orc_e2m1_decode(v) for v in range(16)])
    return table[np.asarray(codes, dtype=np.uint8) & 15]


def e8m0_decode(codes) -> np.ndarray:
    """Values of e8m0 scale bytes, each decoded by the C decoder (a table of its 256 results)."""
    lib = load()
    table = np.array([lib.orc_e8m0_decode(v) for v in range(256)])
    return table[np.asarray(codes, dtype=np.uint8)]


def e2m1_encode(x) -> np.ndarray:
    lib = load()
    a = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_e2m1_encode(float(v)) for v in a], dtype=np.uint8).reshape(np.shape(x))


def quantise_mxfp4_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 rows (reading R23): e2m1 codes [..., c] (one per byte) and e8m0 block
    scales [..., c/32]; decisions in float32."""
    x_ = np.ascontiguousarray(x, dtype=np.float32)
    shp = x_.shape
    c = shp[-1]
    if c % 32:
        raise ValueError("MXFP4 rows need a multiple of 32 values")
    rows = int(np.prod(shp[:-1])) if x_.ndim > 1 else 1
    codes = np.zeros(shp, dtype=np.uint8)
    scales = np.zeros(shp[:-1] + (c // 32,), dtype=np.uint8)
    load().orc_quantise_mxfp4_rows(_ptr(x_), rows, c, _ptr(codes), _ptr(scales))
    return codes, scales


def mxfp4_decode(codes, scales) -> np.ndarray:
    """Values of MXFP4 rows: e2m1(code) * e8m0(scale of its block of 32)."""
    v = e2m1_decode(codes)
    s = e8m0_decode(scales)
    return v * np.repeat(s, 32, axis=-1)
