"""Incremental decode over the heterogeneous KV cache of a hybrid layer pair.

The cache of "DeepSeek-V4 Architecture From Kernels" (shivasnotes.com), section 9:
compressed CSA entries with their FP8 indexer keys, compressed HCA entries, the raw
rows of the blocks not yet complete (the tails), and the exact recent window.
``DecodeSession`` owns that state for one CSA layer and one HCA layer of B sequences
that advance together, allocated once on one device for a capacity of ``n_max``
tokens, and runs one token per ``step``, every stage a library call:

  1. the token's rows go to their ring slots (``token_slots``: a model's projections
     write there directly; ``append`` copies given rows);
  2. when the token completes a CSA block (every m tokens) ``hyb_compress`` pools the
     two blocks the overlapping entry reads, straight from the tail rings, into the
     next entry and its FP8 indexer key; every m' tokens the same for HCA;
  3. ``csa_index_topk`` over the visible entries, ``csa_attend`` of the selected ones
     with the window merged in the same call, then ``hca_attend`` of every visible
     HCA entry with its window ("DeepSeek-V4: Anatomy of an Open-Source Frontier
     Model", "One query in a CSA layer", steps 1-5; "DeepSeek-V4 hybrid attention"
     (trishampatil.com) sections V and VI).

Layout (device, row-major):
  csa_kc [B][N][c], csa_kI [B][N][c_I] e4m3, csa_kIs [B][N] float32, N = n_max / m;
  hca_kc [B][N'][c], N' = n_max / m'.
  CSA tails (ca, cb, za, zb at width c; kIa, kIb, zIa, zIb at width c_I): per sequence
    a ring of 4m rows holding the last 2m tokens twice, token p at slots p mod 2m and
    p mod 2m + 2m.  The 2m rows an overlapping entry pools (blocks i-1 and i) are then
    always consecutive, and the compressor reads them in place, sequences 4m rows apart.
  HCA tails (ch, zh): a ring of m' rows per sequence, token p at slot p mod m' (a block
    starts at slot 0).
  Windows (kv for the CSA layer, kv_h for the HCA layer): 2 n_win rows per sequence,
    token p at slots p mod n_win and p mod n_win + n_win, so that the last n_win
    tokens are consecutive rows; one spare sequence of rows at the end keeps the
    window's view (which starts inside the ring) within the allocation.
"""
from __future__ import annotations

import math

import torch

from . import ops

_CSA_STREAMS = ("ca", "cb", "za", "zb")
_IDX_STREAMS = ("kIa", "kIb", "zIa", "zIb")


class DecodeSession:
    def __init__(self, *, batch: int, n_max: int, n_h: int, c: int, m: int, m_hca: int, k: int, n_ih: int,
                 c_I: int, n_win: int, bias, biasI, bias_h, device, dtype=torch.bfloat16):
        """bias [2m][c], biasI [2m][c_I], bias_h [m'][c]: the compressors' positional biases
        (float32).  n_max: token capacity, a multiple of 4m and of m'."""
        if n_max % (4 * m) or n_max % m_hca:
            raise ValueError("n_max must be a multiple of 4m and of m'")
        self.B, self.n_max, self.n_h, self.c = batch, n_max, n_h, c
        self.m, self.m_hca, self.k, self.n_ih, self.c_I, self.n_win = m, m_hca, k, n_ih, c_I, n_win
        self.dtype, self.device = dtype, torch.device(device)
        self.scale = 1.0 / math.sqrt(c)
        self.bias, self.biasI, self.bias_h = (t.to(self.device, torch.float32).contiguous()
                                              for t in (bias, biasI, bias_h))
        B, dev = batch, self.device
        self.N, self.Nh = n_max // m, n_max // m_hca
        self.csa_kc = torch.zeros((B, self.N, c), dtype=dtype, device=dev)
        self.csa_kI = torch.zeros((B, self.N, c_I), dtype=torch.float8_e4m3fn, device=dev)
        self.csa_kIs = torch.ones((B, self.N), dtype=torch.float32, device=dev)
        self.hca_kc = torch.zeros((B, self.Nh, c), dtype=dtype, device=dev)
        self.tails = {s: torch.zeros((B, 4 * m, c), dtype=dtype, device=dev) for s in _CSA_STREAMS}
        self.tails.update({s: torch.zeros((B, 4 * m, c_I), dtype=dtype, device=dev) for s in _IDX_STREAMS})
        self.tails.update({s: torch.zeros((B, m_hca, c), dtype=dtype, device=dev) for s in ("ch", "zh")})
        # windows: flat rows, sequence b at rows [2 n_win b, 2 n_win (b+1)), one spare sequence
        self.win = {s: torch.zeros(((B + 1) * 2 * n_win, c), dtype=dtype, device=dev) for s in ("kv", "kv_h")}
        self.idx = torch.empty((B, 1, k), dtype=torch.int32, device=dev)
        self.lse = torch.empty((B, 1, n_h), dtype=torch.float32, device=dev)
        self.lse_h = torch.empty((B, 1, n_h), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, 1, n_h, c), dtype=dtype, device=dev)
        self.out_h = torch.empty((B, 1, n_h, c), dtype=dtype, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = {}
        self.t = 0  # position of the next token

    # ------------------------------------------------------------ slots
    @staticmethod
    def csa_slots(p: int, m: int):
        return (p % (2 * m), p % (2 * m) + 2 * m)

    @staticmethod
    def window_slots(p: int, n_win: int):
        return (p % n_win, p % n_win + n_win)

    @staticmethod
    def window_start(t: int, n_win: int):
        """(first ring row of the window view, absolute position of that row) for query t."""
        if t + 1 < n_win:
            return 0, 0
        return (t + 1) % n_win, t - n_win + 1

    @staticmethod
    def csa_block_view(i: int, m: int):
        """Entry i completes: (first ring row, rows, first_block, first entry written)."""
        if i == 0:
            return 0, m, 0, 0
        start = ((i - 1) * m) % (2 * m)
        # with first_block = 0 the call writes entries 0 and 1 (entry 0 again, same values)
        return start, 2 * m, i - 1, (0 if i == 1 else i)

    def token_slots(self, p: int | None = None) -> dict:
        """Where token p's rows go: name -> list of [B, width] views (write each)."""
        p = self.t if p is None else p
        v = {}
        for s in _CSA_STREAMS + _IDX_STREAMS:
            v[s] = [self.tails[s][:, j] for j in self.csa_slots(p, self.m)]
        for s in ("ch", "zh"):
            v[s] = [self.tails[s][:, p % self.m_hca]]
        W = self.n_win
        for s in ("kv", "kv_h"):
            rows = self.win[s][: self.B * 2 * W].view(self.B, 2 * W, self.c)
            v[s] = [rows[:, j] for j in self.window_slots(p, W)]
        return v

    def append(self, rows: dict, p: int | None = None):
        """Copy token p's rows (name -> [B, width]) into their slots."""
        for name, views in self.token_slots(p).items():
            for dst in views:
                dst.copy_(rows[name])

    # ------------------------------------------------------------ state from a prefix
    def prefill(self, chunk: dict, stream=None):
        """Ingest tokens 0..n0-1 (chunk: name -> [B, n0, width]) without computing their
        outputs: compress every complete block into the caches and fill the rings."""
        n0 = chunk["ca"].shape[1]
        if n0 > self.n_max:
            raise ValueError("prefix longer than the session's capacity")
        m, mh, st = self.m, self.m_hca, self.dev_status
        if n0 >= m:
            ops.hyb_compress(chunk["ca"], chunk["za"], self.bias, m, cb=chunk["cb"], zb=chunk["zb"], overlap=True,
                             out=self.csa_kc, out_row0=0, dev_status=st, stream=stream)
            ops.hyb_compress(chunk["kIa"], chunk["zIa"], self.biasI, m, cb=chunk["kIb"], zb=chunk["zIb"],
                             overlap=True, out=self.csa_kI, out_scale=self.csa_kIs, out_row0=0, dev_status=st,
                             stream=stream)
        if n0 >= mh:
            ops.hyb_compress(chunk["ch"], chunk["zh"], self.bias_h, mh, out=self.hca_kc, out_row0=0, dev_status=st,
                             stream=stream)
        self.fill_rings(chunk)

    def fill_rings(self, chunk: dict):
        """The ring part of prefill (no library call): after it the rings hold what
        appending tokens 0..n0-1 one by one leaves in them, and t = n0."""
        n0 = chunk["ca"].shape[1]
        m, mh = self.m, self.m_hca
        # the rings keep what later steps read: the CSA block before the open one and the
        # open one, the open HCA block, the last n_win tokens
        lo = {s: max(0, (n0 // m - 1) * m) for s in _CSA_STREAMS + _IDX_STREAMS}
        lo.update({s: (n0 // mh) * mh for s in ("ch", "zh")})
        lo.update({s: max(0, n0 - self.n_win) for s in ("kv", "kv_h")})
        for s, p0 in lo.items():
            pos = torch.arange(p0, n0, device=self.device)
            if len(pos) == 0:
                continue
            src = chunk[s][:, p0:n0]
            if s in ("kv", "kv_h"):
                W = self.n_win
                rows = self.win[s][: self.B * 2 * W].view(self.B, 2 * W, self.c)
                rows.index_copy_(1, pos % W, src)
                rows.index_copy_(1, pos % W + W, src)
            elif s in ("ch", "zh"):
                self.tails[s].index_copy_(1, pos % mh, src)
            else:
                self.tails[s].index_copy_(1, pos % (2 * m), src)
                self.tails[s].index_copy_(1, pos % (2 * m) + 2 * m, src)
        self.t = n0

    # ------------------------------------------------------------ one token
    def _sizes(self, t):
        """Workspace bytes the calls of a step at position t need."""
        m, mh = self.m, self.m_hca
        dq = lambda *s: torch.empty(s, dtype=self.dtype, device=self.device)
        q1 = dq(self.B, 1, self.n_h, self.c)
        qI1 = torch.empty((self.B, 1, self.n_ih, self.c_I), dtype=torch.float8_e4m3fn, device=self.device)
        f1 = torch.empty((self.B, 1, self.n_ih), dtype=torch.float32, device=self.device)
        a = ops.index_args(qI1, f1, self.csa_kI, m, self.k, t, f1, self.csa_kIs, self.idx, None, (t + 1) // m)
        sizes = {"index": ops.csa_index_topk_workspace_size(a)}
        kw, pos0 = self._window("kv", t)
        a = ops.csa_attend_args(q1, self.csa_kc, self.csa_kc, self.idx, self.scale, None, self.lse, (t + 1) // m,
                                window=ops.window_args(kw, kv_pos0=pos0, q_pos0=t, n_win=self.n_win, out=self.out))
        sizes["csa"] = int(ops._abi.load().csa_attend_workspace_size(a))
        a = ops.hca_attend_args(q1, self.hca_kc, self.hca_kc, mh, t, self.scale, None, self.lse_h, (t + 1) // mh,
                                window=ops.window_args(kw, kv_pos0=pos0, q_pos0=t, n_win=self.n_win, out=self.out_h))
        sizes["hca"] = int(ops._abi.load().hca_attend_workspace_size(a))
        return sizes

    def reserve(self, t_last: int):
        """Allocate the workspaces for every position up to t_last now (for example before
        capturing steps into CUDA graphs, which must not allocate)."""
        for t in {self.t, t_last}:
            for key, n in self._sizes(t).items():
                self._workspace(key, n)

    def _workspace(self, key, nbytes):
        buf = self.ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=self.device)  # counters start at zero
            self.ws[key] = buf
        return buf

    def _window(self, name, t):
        W = self.n_win
        start, pos0 = self.window_start(t, W)
        rows = self.win[name][start:start + self.B * 2 * W]
        return rows.view(self.B, 2 * W, self.c), pos0

    def step(self, *, q, qI, qI_scale, w, q_h, stream=None):
        """Run the layer pair for the token at position t (its rows already appended):
        q, q_h [B, n_h, c]; qI [B, n_ih, c_I] e4m3 with qI_scale [B, n_ih]; w [B, n_ih].
        Returns (out, out_h), [B, 1, n_h, c] each, and advances t."""
        t, m, mh, st = self.t, self.m, self.m_hca, self.dev_status
        if t >= self.n_max:
            raise ValueError("session is full")
        if (t + 1) % m == 0:
            i = (t + 1) // m - 1
            start, rows, fb, row0 = self.csa_block_view(i, m)
            tl = {s: self.tails[s][:, start:start + rows] for s in _CSA_STREAMS + _IDX_STREAMS}
            ops.hyb_compress(tl["ca"], tl["za"], self.bias, m, cb=tl["cb"], zb=tl["zb"], overlap=True,
                             first_block=fb, out=self.csa_kc, out_row0=row0, dev_status=st, stream=stream)
            ops.hyb_compress(tl["kIa"], tl["zIa"], self.biasI, m, cb=tl["kIb"], zb=tl["zIb"], overlap=True,
                             first_block=fb, out=self.csa_kI, out_scale=self.csa_kIs, out_row0=row0, dev_status=st,
                             stream=stream)
        if (t + 1) % mh == 0:
            j = (t + 1) // mh - 1
            ops.hyb_compress(self.tails["ch"], self.tails["zh"], self.bias_h, mh, first_block=j, out=self.hca_kc,
                             out_row0=j, dev_status=st, stream=stream)
        n_vis = (t + 1) // m
        q1, q1h = q.unsqueeze(1), q_h.unsqueeze(1)
        qI1, qIs1, w1 = qI.unsqueeze(1), qI_scale.unsqueeze(1), w.unsqueeze(1)
        a = ops.index_args(qI1, w1, self.csa_kI, m, self.k, t, qIs1, self.csa_kIs, self.idx, None, n_vis)
        ws = self._workspace("index", ops.csa_index_topk_workspace_size(a))
        ops.csa_index_topk(qI1, w1, self.csa_kI, m=m, k=self.k, q_pos0=t, qI_scale=qIs1, kI_scale=self.csa_kIs,
                           n_entries=n_vis, idx=self.idx, workspace=ws, dev_status=st, stream=stream)
        kw, pos0 = self._window("kv", t)
        win = dict(kw=kw, kv_pos0=pos0, q_pos0=t, n_win=self.n_win, out=self.out)
        a = ops.csa_attend_args(q1, self.csa_kc, self.csa_kc, self.idx, self.scale, None, self.lse, n_vis,
                                window=ops.window_args(kw, kv_pos0=pos0, q_pos0=t, n_win=self.n_win, out=self.out))
        ws = self._workspace("csa", int(ops._abi.load().csa_attend_workspace_size(a)))
        ops.csa_attend(q1, self.csa_kc, self.csa_kc, self.idx, scale=self.scale, n_entries=n_vis, lse=self.lse,
                       workspace=ws, dev_status=st, stream=stream, window=win)
        n_vis_h = (t + 1) // mh
        kw, pos0 = self._window("kv_h", t)
        win = dict(kw=kw, kv_pos0=pos0, n_win=self.n_win, out=self.out_h)
        a = ops.hca_attend_args(q1h, self.hca_kc, self.hca_kc, mh, t, self.scale, None, self.lse_h, n_vis_h,
                                window=ops.window_args(kw, kv_pos0=pos0, q_pos0=t, n_win=self.n_win, out=self.out_h))
        ws = self._workspace("hca", int(ops._abi.load().hca_attend_workspace_size(a)))
        ops.hca_attend(q1h, self.hca_kc, self.hca_kc, m=mh, q_pos0=t, scale=self.scale, n_entries=n_vis_h,
                       lse=self.lse_h, workspace=ws, dev_status=st, stream=stream, window=win)
        self.t = t + 1
        return self.out, self.out_h
