"""Torch-facing binding of the C ABI: same names as include/hyb.h.

Each function checks that the tensors it is given are CUDA, dense and of a
dtype the ABI accepts, allocates outputs / workspace with torch when the
caller does not pass them, fills the argument struct and calls the library on
the current (or given) CUDA stream.  No arithmetic of the method happens here:
every step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _abi

# MXFP4 tensors are torch.float4_e2m1fn_x2 (two e2m1 codes per byte: the last dimension counts
# pairs), their scales torch.float8_e8m0fnu (one byte per block of 32 elements)
_DT = {torch.float32: _abi.HYB_F32, torch.bfloat16: _abi.HYB_BF16, torch.float8_e4m3fn: _abi.HYB_E4M3,
       torch.float4_e2m1fn_x2: _abi.HYB_MXFP4}
_TORCH_OF = {v: k for k, v in _DT.items()}


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the hybrid-attention library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the hybrid-attention library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _rows_ptr(t, batch_rows):
    """Pointer of a [B][n][c] view whose rows are contiguous within each sequence and
    whose sequences start batch_rows rows apart (a window of a longer buffer)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the hybrid-attention library must be CUDA tensors")
    B, n, c = t.shape
    if t.stride(2) != 1 or (n > 1 and t.stride(1) != c) or (B > 1 and t.stride(0) != batch_rows * c):
        raise ValueError("compressor inputs: rows must be contiguous, sequences equally spaced")
    return ctypes.c_void_p(t.data_ptr())


def _pos_ptr(t, n, what):
    """Pointer of an int64 device array of n positions (or None)."""
    if t is None:
        return None
    if t.dtype != torch.int64 or t.numel() != n:
        raise ValueError(f"{what} must be int64 with {n} elements")
    return _ptr(t)


def _dtype(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, workspace, device, zeroed=False):
    """zeroed: the call needs the workspace to start zero-filled (csa_index_topk, csa_attend
    and hca_attend keep counters in its first bytes and leave them zero); a caller's own
    workspace must then have been zero-filled once."""
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = (torch.zeros if zeroed else torch.empty)(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, {nbytes} needed")
    return _ptr(workspace), workspace.numel() * workspace.element_size()


# ------------------------------------------------------------------ compress


def compress_out_count(n_rows: int, m: int, overlap: bool, first_block: int = 0) -> int:
    return int(_abi.load().hyb_compress_out_count(n_rows, m, int(bool(overlap)), first_block))


def compress_args(ca, za, bias, m, cb=None, zb=None, overlap=False, first_block=0, out=None, out_scale=None,
                  out_batch_stride=0, out_dtype=None, dev_status=None, out_row0=0):
    """Argument struct of hyb_compress.  The entries are written from row out_row0 of
    out ([B][rows][c]) on; the batch stride is out's row count."""
    B, n, c = ca.shape
    # the inputs may be windows of longer per-sequence buffers (all with the same spacing)
    rows = ca.stride(0) // c if B > 1 else n
    a = _abi.CompressArgs()
    a.ca, a.cb, a.za, a.zb = (_rows_ptr(t, rows) for t in (ca, cb, za, zb))
    a.bias = _ptr(bias)
    a.in_batch_stride = 0 if rows == n else rows
    a.out, a.out_scale = _ptr(out), _ptr(out_scale)
    if out is not None:
        if out_row0:  # (row strides of out and out_scale: c values or c/2 pairs; one scale or c/32)
            a.out = ctypes.c_void_p(out.data_ptr() + out_row0 * out.stride(1) * out.element_size())
            if out_scale is not None:
                rs = out_scale.stride(1) if out_scale.dim() == 3 else 1
                a.out_scale = ctypes.c_void_p(out_scale.data_ptr() + out_row0 * rs * out_scale.element_size())
        out_batch_stride = out.shape[1]
    a.batch, a.n_rows, a.c, a.m, a.first_block = B, n, c, m, first_block
    a.out_batch_stride = out_batch_stride
    a.overlap = int(bool(overlap))
    a.in_dtype = _dtype(ca)
    a.out_dtype = _dtype(out) if out is not None else _DT[out_dtype]
    a.dev_status = _ptr(dev_status)
    return a


def hyb_compress(ca, za, bias, m: int, *, cb=None, zb=None, overlap: bool = False, first_block: int = 0,
                 out=None, out_scale=None, out_dtype=None, out_batch_stride: int = 0, out_row0: int = 0,
                 dev_status=None, stream=None):
    """Softmax-gated compressor.  Returns (out, out_scale or None).

    out_row0 writes the entries into rows out_row0.. of an existing [B][rows][c]
    buffer (a cache slot in decode)."""
    B, n, c = ca.shape
    n_out = compress_out_count(n, m, overlap, first_block)
    if out is None:
        dt = out_dtype if out_dtype is not None else ca.dtype
        if dt == torch.float4_e2m1fn_x2:
            out = torch.empty((B, n_out, c // 2), dtype=dt, device=ca.device)
            if out_scale is None:
                out_scale = torch.empty((B, n_out, c // 32), dtype=torch.float8_e8m0fnu, device=ca.device)
        else:
            out = torch.empty((B, n_out, c), dtype=dt, device=ca.device)
        if dt == torch.float8_e4m3fn and out_scale is None:
            out_scale = torch.empty((B, n_out), dtype=torch.float32, device=ca.device)
    if out_row0 and (out_row0 + n_out > out.shape[1]):
        raise ValueError("out_row0 + entries exceeds the rows of out")
    a = compress_args(ca, za, bias, m, cb, zb, overlap, first_block, out, out_scale, out_batch_stride, None,
                      dev_status, out_row0)
    lib = _abi.load()
    _abi.check(lib.hyb_compress(ctypes.byref(a), None, 0, _stream(stream)), "hyb_compress")
    return out, out_scale


def compress_call(a, stream=None):
    """hyb_compress on an argument struct from compress_args."""
    _abi.check(_abi.load().hyb_compress(ctypes.byref(a), None, 0, _stream(stream)), "hyb_compress")


def hyb_compress_batch(calls, stream=None):
    """Several compressions in one launch (hyb_compress_batch): calls is a list of argument
    structs from compress_args (each with its out given), at most HYB_COMPRESS_BATCH_MAX."""
    arr = (_abi.CompressArgs * max(1, len(calls)))(*calls)
    _abi.check(_abi.load().hyb_compress_batch(arr, len(calls), _stream(stream)), "hyb_compress_batch")


# ------------------------------------------------------------- index + top-k


def index_args(qI, w, kI, m, k, q_pos0, qI_scale=None, kI_scale=None, idx=None, scores=None, n_entries=None,
               dev_status=None, scores_events=None, q_pos=None):
    """q_pos: optional int64 [B, n_q] per-query absolute positions (then q_pos0 is unused).
    MXFP4 (qI, kI float4_e2m1fn_x2, last dimension c_I/2; scales float8_e8m0fnu [..., c_I/32])."""
    B, n_q, n_ih, c_I = qI.shape
    if qI.dtype == torch.float4_e2m1fn_x2:
        c_I *= 2
    a = _abi.IndexArgs()
    a.qI, a.qI_scale, a.w, a.kI, a.kI_scale = _ptr(qI), _ptr(qI_scale), _ptr(w), _ptr(kI), _ptr(kI_scale)
    a.idx, a.scores = _ptr(idx), _ptr(scores)
    a.batch, a.n_q, a.n_ih, a.c_I, a.m, a.k, a.q_pos0 = B, n_q, n_ih, c_I, m, k, q_pos0
    a.n_entries = kI.shape[1] if n_entries is None else n_entries
    a.kv_stride = kI.shape[1]
    a.dtype = _dtype(qI)
    a.dev_status = _ptr(dev_status)
    if scores_events is not None:  # (begin, end) torch.cuda.Event: recorded around the scoring kernel
        a.ev_scores_begin, a.ev_scores_end = (ctypes.c_void_p(int(e.cuda_event)) for e in scores_events)
    a.q_pos = _pos_ptr(q_pos, B * n_q, "q_pos")
    return a


def csa_index_topk_workspace_size(a) -> int:
    return int(_abi.load().csa_index_topk_workspace_size(ctypes.byref(a)))


def csa_index_topk_counter_bytes() -> int:
    """Leading bytes of a csa_index_topk workspace that must be zero before a call
    (every call leaves them zero; re-zero them after a device timeout)."""
    return int(_abi.load().csa_index_topk_counter_bytes())


def csa_index_topk(qI, w, kI, *, m: int, k: int, q_pos0: int = 0, qI_scale=None, kI_scale=None, n_entries=None,
                   idx=None, scores=None, want_scores: bool = False, workspace=None, dev_status=None, stream=None,
                   scores_events=None, q_pos=None):
    """Lightning-indexer scores + top-k.  Returns idx (and the selected scores when asked).
    scores_events: optional (begin, end) torch.cuda.Event, recorded around the scoring kernel.
    q_pos: optional int64 [B, n_q] per-query positions (instead of q_pos0 + j)."""
    B, n_q = qI.shape[:2]
    if idx is None:
        idx = torch.empty((B, n_q, k), dtype=torch.int32, device=qI.device)
    if scores is None and want_scores:
        scores = torch.empty((B, n_q, k), dtype=torch.float32, device=qI.device)
    a = index_args(qI, w, kI, m, k, q_pos0, qI_scale, kI_scale, idx, scores, n_entries, dev_status, scores_events,
                   q_pos)
    ws, nbytes = _workspace(csa_index_topk_workspace_size(a), workspace, qI.device, zeroed=True)
    _abi.check(_abi.load().csa_index_topk(ctypes.byref(a), ws, nbytes, _stream(stream)), "csa_index_topk")
    return (idx, scores) if want_scores else idx


# ---------------------------------------------------------------- attention


def window_args(kw, *, kv_pos0: int = 0, q_pos0: int = 0, n_win: int, out, q_pos=None, kv_pos0s=None):
    """The fused window merge of csa_attend / hca_attend (hyb_window): the raw rows kw
    [B, n_kv, c] (row 0 = absolute position kv_pos0, or kv_pos0s[b] per sequence) are the
    window's keys and values; out [B, n_q, n_h, c] receives the merged output.  q_pos:
    optional int64 [B, n_q] per-query positions; kv_pos0s: optional int64 [B]."""
    w = _abi.Window()
    w.kw, w.n_kv, w.kv_pos0, w.q_pos0, w.n_win = _ptr(kw), kw.shape[1], kv_pos0, q_pos0, n_win
    w.out, w.out_dtype = _ptr(out), _dtype(out)
    B, n_q = out.shape[:2]
    w.q_pos = _pos_ptr(q_pos, B * n_q, "window q_pos")
    w.kv_pos0s = _pos_ptr(kv_pos0s, B, "window kv_pos0s")
    return w


def _check_sink(sink, n_h):
    if sink is not None and (sink.dtype != torch.float32 or sink.numel() != n_h):
        raise ValueError("sink must be float32 [n_h]")


def csa_attend_args(q, kc, vc, idx, scale, o, lse, n_entries=None, dev_status=None, window=None, sink=None):
    B, n_q, n_h, c = q.shape
    _check_sink(sink, n_h)
    a = _abi.CsaAttendArgs()
    a.q, a.kc, a.vc, a.idx, a.o, a.lse = _ptr(q), _ptr(kc), _ptr(vc), _ptr(idx), _ptr(o), _ptr(lse)
    a.batch, a.n_q, a.n_h, a.c = B, n_q, n_h, c
    a.n_entries = kc.shape[1] if n_entries is None else n_entries
    a.kv_stride = kc.shape[1]
    a.k = idx.shape[-1]
    a.scale = scale
    a.dtype = _dtype(q)
    a.dev_status = _ptr(dev_status)
    a._window = window  # keep the struct alive as long as the arguments
    a.window = ctypes.cast(ctypes.pointer(window), ctypes.c_void_p) if window is not None else None
    a.sink = _ptr(sink)
    return a


def _window(q, window):
    """window: None or dict(kw=, kv_pos0=, q_pos0=, n_win=, out= (optional), out_dtype= (optional))."""
    if window is None:
        return None, None
    w = dict(window)
    out = w.pop("out", None)
    if out is None:
        B, n_q, n_h, c = q.shape
        out = torch.empty((B, n_q, n_h, c), dtype=w.pop("out_dtype", None) or q.dtype, device=q.device)
    w.pop("out_dtype", None)
    return window_args(w.pop("kw"), out=out, **w), out


def csa_attend(q, kc, vc, idx, *, scale: float | None = None, n_entries=None, o=None, lse=None, workspace=None,
               dev_status=None, stream=None, window=None, sink=None):
    """CSA core attention over the selected entries.  Returns (o, lse), or (out, lse) of the
    union with a fused window merge (window=dict(kw, kv_pos0, q_pos0, n_win[, out])).
    sink: optional float32 [n_h] per-head attention-sink logits, applied to the result."""
    B, n_q, n_h, c = q.shape
    scale = 1.0 / math.sqrt(c) if scale is None else scale
    w, out = _window(q, window)
    if o is None and w is None:
        o = torch.empty((B, n_q, n_h, c), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, n_q, n_h), dtype=torch.float32, device=q.device) if lse is None else lse
    a = csa_attend_args(q, kc, vc, idx, scale, o, lse, n_entries, dev_status, w, sink)
    lib = _abi.load()
    ws, nbytes = _workspace(int(lib.csa_attend_workspace_size(ctypes.byref(a))), workspace, q.device, zeroed=True)
    _abi.check(lib.csa_attend(ctypes.byref(a), ws, nbytes, _stream(stream)), "csa_attend")
    return (out, lse) if w is not None else (o, lse)


def hca_attend_args(q, kc, vc, m, q_pos0, scale, o, lse, n_entries=None, dev_status=None, window=None, sink=None,
                    q_pos=None):
    B, n_q, n_h, c = q.shape
    _check_sink(sink, n_h)
    a = _abi.HcaAttendArgs()
    a.q, a.kc, a.vc, a.o, a.lse = _ptr(q), _ptr(kc), _ptr(vc), _ptr(o), _ptr(lse)
    a.batch, a.n_q, a.n_h, a.c = B, n_q, n_h, c
    a.n_entries = kc.shape[1] if n_entries is None else n_entries
    a.kv_stride = kc.shape[1]
    a.m, a.q_pos0, a.scale = m, q_pos0, scale
    a.dtype = _dtype(q)
    a.dev_status = _ptr(dev_status)
    a._window = window
    a.window = ctypes.cast(ctypes.pointer(window), ctypes.c_void_p) if window is not None else None
    a.sink = _ptr(sink)
    a.q_pos = _pos_ptr(q_pos, B * n_q, "q_pos")
    return a


def hca_attend(q, kc, vc, *, m: int, q_pos0: int = 0, scale: float | None = None, n_entries=None, o=None,
               lse=None, workspace=None, dev_status=None, stream=None, window=None, sink=None, q_pos=None):
    """HCA core attention over every visible entry.  Returns (o, lse), or (out, lse) of the
    union with a fused window merge (window=dict(kw, kv_pos0 or kv_pos0s, n_win[, out]); the
    window's query positions are the call's).  sink: optional float32 [n_h] per-head
    attention-sink logits, applied to the result.  q_pos: optional int64 [B, n_q] per-query
    positions (instead of q_pos0 + j)."""
    B, n_q, n_h, c = q.shape
    scale = 1.0 / math.sqrt(c) if scale is None else scale
    if window is not None:
        window = dict(window, q_pos0=q_pos0, q_pos=q_pos)
    w, out = _window(q, window)
    if o is None and w is None:
        o = torch.empty((B, n_q, n_h, c), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, n_q, n_h), dtype=torch.float32, device=q.device) if lse is None else lse
    a = hca_attend_args(q, kc, vc, m, q_pos0, scale, o, lse, n_entries, dev_status, w, sink, q_pos)
    lib = _abi.load()
    ws, nbytes = _workspace(int(lib.hca_attend_workspace_size(ctypes.byref(a))), workspace, q.device, zeroed=True)
    _abi.check(lib.hca_attend(ctypes.byref(a), ws, nbytes, _stream(stream)), "hca_attend")
    return (out, lse) if w is not None else (o, lse)


def swa_args(q, kw, vw, kv_pos0, q_pos0, n_win, scale, o_in, lse_in, out, lse_out, dev_status=None, q_pos=None,
             kv_pos0s=None):
    B, n_q, n_h, c = q.shape
    a = _abi.SwaArgs()
    a.q, a.kw, a.vw, a.o_in, a.lse_in, a.out, a.lse_out = (_ptr(q), _ptr(kw), _ptr(vw), _ptr(o_in), _ptr(lse_in),
                                                           _ptr(out), _ptr(lse_out))
    a.batch, a.n_q, a.n_h, a.c = B, n_q, n_h, c
    a.n_kv, a.kv_pos0, a.q_pos0, a.n_win, a.scale = kw.shape[1], kv_pos0, q_pos0, n_win, scale
    a.dtype = _dtype(q)
    a.out_dtype = _dtype(out)
    a.dev_status = _ptr(dev_status)
    a.q_pos = _pos_ptr(q_pos, B * n_q, "q_pos")
    a.kv_pos0s = _pos_ptr(kv_pos0s, B, "kv_pos0s")
    return a


def swa_merge(q, kw, vw, *, kv_pos0: int = 0, q_pos0: int = 0, n_win: int, scale: float | None = None, o_in=None,
              lse_in=None, out=None, out_dtype=None, lse_out=None, want_lse: bool = False, workspace=None,
              dev_status=None, stream=None, q_pos=None, kv_pos0s=None):
    """Sliding-window branch merged with (o_in, lse_in) by log-sum-exp.  Returns out (and lse when asked).
    q_pos: optional int64 [B, n_q] per-query positions; kv_pos0s: optional int64 [B] per-sequence
    absolute position of row 0 of kw / vw."""
    B, n_q, n_h, c = q.shape
    scale = 1.0 / math.sqrt(c) if scale is None else scale
    if out is None:
        out = torch.empty((B, n_q, n_h, c), dtype=out_dtype or q.dtype, device=q.device)
    if lse_out is None and want_lse:
        lse_out = torch.empty((B, n_q, n_h), dtype=torch.float32, device=q.device)
    a = swa_args(q, kw, vw, kv_pos0, q_pos0, n_win, scale, o_in, lse_in, out, lse_out, dev_status, q_pos, kv_pos0s)
    lib = _abi.load()
    ws, nbytes = _workspace(int(lib.swa_merge_workspace_size(ctypes.byref(a))), workspace, q.device)
    _abi.check(lib.swa_merge(ctypes.byref(a), ws, nbytes, _stream(stream)), "swa_merge")
    return (out, lse_out) if want_lse else out


# ------------------------------------------------------------ RMSNorm + RoPE


def rmsnorm_rope_args(x, *, gamma=None, eps: float = 1e-6, pos=None, rows_per_pos: int = 1, rope_dims: int = 64,
                      theta: float = 10000.0):
    """Argument struct of hyb_rmsnorm_rope for x (see rmsnorm_rope)."""
    c = x.shape[-1]
    rows = x.numel() // c
    row_stride = 0
    if not x.is_contiguous():
        if x.dim() != 2 or x.stride(1) != 1 or x.stride(0) < c:
            raise ValueError("x must be contiguous or a [rows, c] view with unit column stride")
        row_stride = x.stride(0)
    if pos is not None and (pos.dtype != torch.int64 or pos.numel() * rows_per_pos < rows):
        raise ValueError("pos must be int64 with one position per rows_per_pos rows")
    if gamma is not None and (gamma.dtype != torch.float32 or gamma.numel() != c):
        raise ValueError("gamma must be float32 [c]")
    a = _abi.NormRopeArgs()
    if not x.is_cuda:
        raise ValueError("tensors passed to the hybrid-attention library must be CUDA tensors")
    a.x, a.rows, a.c = ctypes.c_void_p(x.data_ptr()), rows, c
    a.gamma, a.eps, a.dtype = _ptr(gamma), eps, _dtype(x)
    a.pos, a.rows_per_pos = _ptr(pos), rows_per_pos
    a.rope_dims, a.theta = (rope_dims if pos is not None else 0), theta
    a.row_stride = row_stride
    return a


def rmsnorm_rope(x, *, gamma=None, eps: float = 1e-6, pos=None, rows_per_pos: int = 1, rope_dims: int = 64,
                 theta: float = 10000.0, stream=None):
    """In place: RMSNorm of every row of x [..., c] (float32 or bf16), then rotary
    encoding of its last rope_dims dimensions at positions pos (int64, one per
    rows_per_pos consecutive rows; rope_dims=0 or pos=None: no rotation).  x is
    contiguous, or a 2-D view [rows, c] of unit column stride whose rows are evenly
    spaced (e.g. one cache slot of every sequence).  Returns x."""
    a = rmsnorm_rope_args(x, gamma=gamma, eps=eps, pos=pos, rows_per_pos=rows_per_pos, rope_dims=rope_dims,
                          theta=theta)
    _abi.check(_abi.load().hyb_rmsnorm_rope(ctypes.byref(a), _stream(stream)), "hyb_rmsnorm_rope")
    return x


def rmsnorm_rope_batch(calls, stream=None):
    """Several RMSNorm + RoPE calls of one dtype in one launch (hyb_rmsnorm_rope_batch):
    calls is a list of argument structs from rmsnorm_rope_args, at most
    HYB_NORM_ROPE_BATCH_MAX."""
    arr = (_abi.NormRopeArgs * max(1, len(calls)))(*calls)
    _abi.check(_abi.load().hyb_rmsnorm_rope_batch(arr, len(calls), _stream(stream)), "hyb_rmsnorm_rope_batch")


# ---------------------------------------------------- grouped output projection


def grouped_out_proj(o, w, *, out=None, out_dtype=torch.float32, dev_status=None, stream=None):
    """Grouped output projection: o [..., n_h, c] bf16 (the heads of each row), w [g, d_g,
    (n_h/g)*c] bf16.  Returns out [..., g*d_g] (out_dtype float32 or bf16): group j of n_h/g
    consecutive heads projected by w[j], the g results concatenated.  out may be a column
    slice of a wider [rows, F] buffer (rows contiguous, row stride F): the call then fills
    its g*d_g columns."""
    n_h, c = o.shape[-2], o.shape[-1]
    g, d_g, k = w.shape
    if k * g != n_h * c:
        raise ValueError("w must be [g, d_g, (n_h/g)*c]")
    lead = o.shape[:-2]
    rows = math.prod(lead) if lead else 1
    if out is None:
        out = torch.empty(tuple(lead) + (g * d_g,), dtype=out_dtype, device=o.device)
    if out.shape[-1] != g * d_g or out.stride(-1) != 1:
        raise ValueError("out must end in g*d_g contiguous features")
    a = _abi.GprojArgs()
    a.o, a.w = _ptr(o), _ptr(w)
    if not out.is_cuda:
        raise ValueError("tensors passed to the hybrid-attention library must be CUDA tensors")
    a.out = ctypes.c_void_p(out.data_ptr())
    a.out_row_stride = out.stride(-2) if out.dim() >= 2 and rows > 1 else 0
    a.rows, a.n_h, a.c, a.g, a.d_g = rows, n_h, c, g, d_g
    a.dtype, a.out_dtype = _dtype(o), _dtype(out)
    if _dtype(w) != a.dtype:
        raise ValueError("o and w must have the same dtype")
    a.dev_status = _ptr(dev_status)
    _abi.check(_abi.load().hyb_grouped_out_proj(ctypes.byref(a), _stream(stream)), "hyb_grouped_out_proj")
    return out
