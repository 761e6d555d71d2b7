"""Incremental decode over the heterogeneous KV cache of a hybrid layer pair.

The cache of "DeepSeek-V4 Architecture From Kernels" (shivasnotes.com), section 9:
compressed CSA entries with their FP8 indexer keys, compressed HCA entries, the raw
rows of the blocks not yet complete (the tails), and the exact recent window.
``DecodeSession`` owns that state for one CSA layer and one HCA layer of B sequences,
allocated once on one device for a capacity of ``n_max`` tokens, and runs one token
per sequence per ``step``, every stage a library call.  The sequences may sit at
different lengths (a prefix of its own length each): they then carry per-sequence
positions, which the calls take as device arrays (``q_pos``, and ``kv_pos0s`` for
the windows read in place from each sequence's ring).

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
  Rings, packed by width: rings [9][B][R][c] (ca, cb, za, zb, ch, zh, kv, kv_h and a
  spare), R = max(4m, m', 2 n_win); rings_I [4][B][4m][c_I] (kIa, kIb, zIa, zIb).
  CSA tails (ca, cb, za, zb; kIa, kIb, zIa, zIb): the last 2m tokens twice, token p at
    slots p mod 2m and p mod 2m + 2m.  The 2m rows an overlapping entry pools (blocks
    i-1 and i) are then always consecutive, and the compressor reads them in place
    (sequences R rows apart).
  HCA tails (ch, zh): token p at slot p mod m' (a block starts at slot 0).
  Windows (kv for the CSA layer, kv_h for the HCA layer): token p at slots p mod n_win
    and p mod n_win + n_win, so that the last n_win tokens are consecutive rows; the
    window's view starts inside its ring and may run into the next one (hence the
    spare ring), never past the allocation.
  A token's rows land with one gather and one scatter per width (slot table on the
  device, indexed by the position modulo the rings' common period).
"""
from __future__ import annotations

import math

import torch

from . import ops

_CSA_STREAMS = ("ca", "cb", "za", "zb")
_IDX_STREAMS = ("kIa", "kIb", "zIa", "zIb")
_WIDE = _CSA_STREAMS + ("ch", "zh", "kv", "kv_h")  # width c, ring order in `rings`


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
        self.R = max(4 * m, m_hca, 2 * n_win)
        self.rings = torch.zeros((len(_WIDE) + 1, B, self.R, c), dtype=dtype, device=dev)
        self.rings_I = torch.zeros((len(_IDX_STREAMS), B, 4 * m, c_I), dtype=dtype, device=dev)
        # the writes of one token: (ring, slot) per write, slots tabulated over the period
        self.period = math.lcm(2 * m, m_hca, n_win)
        self._writes, self._writes_I = [], []
        for s in _WIDE:
            for j in range(1 if s in ("ch", "zh") else 2):
                self._writes.append((s, j))
        for s in _IDX_STREAMS:
            for j in range(2):
                self._writes_I.append((s, j))
        ring_ids = lambda ws, order: torch.tensor([order.index(s) for s, _ in ws], dtype=torch.long, device=dev)
        self._ring_ids = ring_ids(self._writes, _WIDE)
        self._ring_ids_I = ring_ids(self._writes_I, _IDX_STREAMS)
        self._slot_tab = torch.tensor([[self._slot(s, j, p) for s, j in self._writes] for p in range(self.period)],
                                      dtype=torch.long, device=dev)
        self._slot_tab_I = torch.tensor([[self._slot(s, j, p) for s, j in self._writes_I]
                                         for p in range(self.period)], dtype=torch.long, device=dev)
        self.idx = torch.empty((B, 1, k), dtype=torch.int32, device=dev)
        self.lse = torch.empty((B, 1, n_h), dtype=torch.float32, device=dev)
        self.lse_h = torch.empty((B, 1, n_h), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, 1, n_h, c), dtype=dtype, device=dev)
        self.out_h = torch.empty((B, 1, n_h, c), dtype=dtype, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = {}
        self.tb = [0] * B  # position of each sequence's next token
        self.pos = torch.zeros(B, dtype=torch.int64, device=dev)  # the same, on the device (ragged steps)

    @property
    def t(self) -> int:
        """Position of the next token when every sequence is at the same one."""
        if any(x != self.tb[0] for x in self.tb):
            raise ValueError("the sequences sit at different positions: see tb")
        return self.tb[0]

    @t.setter
    def t(self, value: int):
        # (the device copy `pos` is used only by ragged steps, which keep it themselves)
        self.tb = [int(value)] * self.B

    @property
    def ragged(self) -> bool:
        return any(x != self.tb[0] for x in self.tb)

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

    def _slot(self, name, j, p):
        """Ring slot of copy j of token p's row of stream `name`."""
        if name in ("ch", "zh"):
            return p % self.m_hca
        if name in ("kv", "kv_h"):
            return self.window_slots(p, self.n_win)[j]
        return self.csa_slots(p, self.m)[j]

    def ring(self, name) -> torch.Tensor:
        """The ring of a stream: [B][R][c] (or [B][4m][c_I] for the indexer-key streams)."""
        if name in _IDX_STREAMS:
            return self.rings_I[_IDX_STREAMS.index(name)]
        return self.rings[_WIDE.index(name)]

    def token_slots(self, p: int | None = None) -> dict:
        """Where token p's rows go: name -> list of [B, width] views (write each)."""
        p = self.t if p is None else p
        v = {}
        for s, j in self._writes + self._writes_I:
            v.setdefault(s, []).append(self.ring(s)[:, self._slot(s, j, p)])
        return v

    def append(self, rows: dict, p: int | None = None):
        """Put the next token's rows (name -> [B, width]) into their slots: per width, one
        gather of the rows and one scatter into the rings.  p: the position, when every
        sequence is at the same one (default: each sequence's own next position)."""
        if p is None and self.ragged:
            # per-sequence slots, looked up on the device from the sequences' positions
            k = self.pos % self.period
            bi = torch.arange(self.B, device=self.device).view(1, -1)
            self.rings[self._ring_ids.view(-1, 1), bi, self._slot_tab[k].T] = \
                torch.stack([rows[s] for s, _ in self._writes])
            self.rings_I[self._ring_ids_I.view(-1, 1), bi, self._slot_tab_I[k].T] = \
                torch.stack([rows[s] for s, _ in self._writes_I])
            return
        p = self.t if p is None else p
        k = p % self.period
        self.rings[self._ring_ids, :, self._slot_tab[k]] = torch.stack([rows[s] for s, _ in self._writes])
        self.rings_I[self._ring_ids_I, :, self._slot_tab_I[k]] = torch.stack([rows[s] for s, _ in self._writes_I])

    # ------------------------------------------------------------ state from a prefix
    def prefill(self, chunk: dict, stream=None, lengths=None):
        """Ingest tokens 0..n0-1 (chunk: name -> [B, n0, width]) without computing their
        outputs: compress every complete block into the caches and fill the rings.
        lengths: optional per-sequence prefix lengths (<= n0): sequence b keeps only its
        first lengths[b] tokens (entries of blocks past them are never visible to it
        and are rewritten when its own tokens complete them)."""
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
        if lengths is None:
            self.fill_rings(chunk)
            return
        for b, n in enumerate(lengths):
            if not 0 <= n <= n0:
                raise ValueError("each prefix length must be within the chunk")
            self._fill_rings_of(b, {k: v[b:b + 1, :n] for k, v in chunk.items()})
        self.tb = [int(n) for n in lengths]
        self.pos.copy_(torch.tensor(self.tb, dtype=torch.int64))

    def fill_rings(self, chunk: dict):
        """The ring part of prefill (no library call): after it the rings hold what
        appending tokens 0..n0-1 one by one leaves in them, and t = n0."""
        self._fill_rings_of(None, chunk)
        self.t = chunk["ca"].shape[1]

    def _fill_rings_of(self, b, chunk: dict):
        """Rings of sequence b (every sequence when b is None) from its tokens 0..n0-1."""
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
            src, r = chunk[s][:, p0:n0], self.ring(s)
            if b is not None:
                r = r[b:b + 1]
            if s in ("kv", "kv_h"):
                W = self.n_win
                r.index_copy_(1, pos % W, src)
                r.index_copy_(1, pos % W + W, src)
            elif s in ("ch", "zh"):
                r.index_copy_(1, pos % mh, src)
            else:
                r.index_copy_(1, pos % (2 * m), src)
                r.index_copy_(1, pos % (2 * m) + 2 * m, src)

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
        """The window of query t as [B][R][c] rows (row 0 at the returned position), a
        view that starts inside the stream's ring."""
        start, pos0 = self.window_start(t, self.n_win)
        first = _WIDE.index(name) * self.B * self.R + start
        rows = self.rings.view(-1, self.c)[first:first + self.B * self.R]
        return rows.view(self.B, self.R, self.c), pos0

    def step(self, *, q, qI, qI_scale, w, q_h, stream=None):
        """Run the layer pair for each sequence's token at its position (its rows already
        appended): q, q_h [B, n_h, c]; qI [B, n_ih, c_I] e4m3 with qI_scale [B, n_ih];
        w [B, n_ih].  Returns (out, out_h), [B, 1, n_h, c] each, and advances the positions."""
        if self.ragged:
            return self._step_ragged(q=q, qI=qI, qI_scale=qI_scale, w=w, q_h=q_h, stream=stream)
        t, m, mh, st = self.t, self.m, self.m_hca, self.dev_status
        if t >= self.n_max:
            raise ValueError("session is full")
        calls = []  # the entries this token completes, compressed in one launch
        if (t + 1) % m == 0:
            i = (t + 1) // m - 1
            start, rows, fb, row0 = self.csa_block_view(i, m)
            tl = {s: self.ring(s)[:, start:start + rows] for s in _CSA_STREAMS + _IDX_STREAMS}
            calls.append(ops.compress_args(tl["ca"], tl["za"], self.bias, m, tl["cb"], tl["zb"], True, fb, self.csa_kc,
                                           None, dev_status=st, out_row0=row0))
            calls.append(ops.compress_args(tl["kIa"], tl["zIa"], self.biasI, m, tl["kIb"], tl["zIb"], True, fb,
                                           self.csa_kI, self.csa_kIs, dev_status=st, out_row0=row0))
        if (t + 1) % mh == 0:
            j = (t + 1) // mh - 1
            calls.append(ops.compress_args(self.ring("ch")[:, :mh], self.ring("zh")[:, :mh], self.bias_h, mh,
                                           first_block=j, out=self.hca_kc, dev_status=st, out_row0=j))
        if len(calls) == 3:  # both layers: one launch (slower than two launches for the CSA pair alone)
            ops.hyb_compress_batch(calls, stream=stream)
        else:
            for a in calls:
                ops.compress_call(a, stream=stream)
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

    def _step_ragged(self, *, q, qI, qI_scale, w, q_h, stream=None):
        """step() for sequences at different positions: each sequence that completes a
        block compresses its own entry (a call on that sequence's rows alone); the
        indexer and both attentions run once over the batch with per-sequence positions
        (q_pos), the windows read in place from each sequence's ring (kv_pos0s)."""
        m, mh, st, W = self.m, self.m_hca, self.dev_status, self.n_win
        if max(self.tb) >= self.n_max:
            raise ValueError("session is full")
        for b, t in enumerate(self.tb):
            sl = slice(b, b + 1)
            if (t + 1) % m == 0:
                start, rows, fb, row0 = self.csa_block_view((t + 1) // m - 1, m)
                tl = {s: self.ring(s)[sl, start:start + rows] for s in _CSA_STREAMS + _IDX_STREAMS}
                ops.hyb_compress(tl["ca"], tl["za"], self.bias, m, cb=tl["cb"], zb=tl["zb"], overlap=True,
                                 first_block=fb, out=self.csa_kc[sl], out_row0=row0, dev_status=st, stream=stream)
                ops.hyb_compress(tl["kIa"], tl["zIa"], self.biasI, m, cb=tl["kIb"], zb=tl["zIb"], overlap=True,
                                 first_block=fb, out=self.csa_kI[sl], out_scale=self.csa_kIs[sl], out_row0=row0,
                                 dev_status=st, stream=stream)
            if (t + 1) % mh == 0:
                j = (t + 1) // mh - 1
                ops.hyb_compress(self.ring("ch")[sl, :mh], self.ring("zh")[sl, :mh], self.bias_h, mh, first_block=j,
                                 out=self.hca_kc[sl], out_row0=j, dev_status=st, stream=stream)
        q_pos = self.pos.view(self.B, 1)
        # row 0 of each sequence's window ring holds the first position of the period the
        # window starts in (token p sits at rows p mod W and p mod W + W)
        kv_pos0s = (self.pos - (W - 1)).clamp_(min=0).div_(W, rounding_mode="floor").mul_(W)
        q1, q1h = q.unsqueeze(1), q_h.unsqueeze(1)
        qI1, qIs1, w1 = qI.unsqueeze(1), qI_scale.unsqueeze(1), w.unsqueeze(1)
        a = ops.index_args(qI1, w1, self.csa_kI, m, self.k, 0, qIs1, self.csa_kIs, self.idx, None, q_pos=q_pos)
        ws = self._workspace("index_r", ops.csa_index_topk_workspace_size(a))
        ops.csa_index_topk(qI1, w1, self.csa_kI, m=m, k=self.k, q_pos=q_pos, qI_scale=qIs1, kI_scale=self.csa_kIs,
                           idx=self.idx, workspace=ws, dev_status=st, stream=stream)
        kw = self.ring("kv")
        win = dict(kw=kw, q_pos=q_pos, kv_pos0s=kv_pos0s, n_win=W, out=self.out)
        a = ops.csa_attend_args(q1, self.csa_kc, self.csa_kc, self.idx, self.scale, None, self.lse,
                                window=ops.window_args(**win))
        ws = self._workspace("csa_r", int(ops._abi.load().csa_attend_workspace_size(a)))
        ops.csa_attend(q1, self.csa_kc, self.csa_kc, self.idx, scale=self.scale, lse=self.lse, workspace=ws,
                       dev_status=st, stream=stream, window=win)
        win = dict(kw=self.ring("kv_h"), kv_pos0s=kv_pos0s, n_win=W, out=self.out_h)
        a = ops.hca_attend_args(q1h, self.hca_kc, self.hca_kc, mh, 0, self.scale, None, self.lse_h,
                                window=ops.window_args(**win, q_pos=q_pos), q_pos=q_pos)
        ws = self._workspace("hca_r", int(ops._abi.load().hca_attend_workspace_size(a)))
        ops.hca_attend(q1h, self.hca_kc, self.hca_kc, m=mh, q_pos=q_pos, scale=self.scale, lse=self.lse_h,
                       workspace=ws, dev_status=st, stream=stream, window=win)
        self.tb = [t + 1 for t in self.tb]
        self.pos.add_(1)
        return self.out, self.out_h
