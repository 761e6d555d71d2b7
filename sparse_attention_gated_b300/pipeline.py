"""One forward step of a hybrid-attention workload, every stage a library call.

``HybridStep`` owns the output buffers and workspaces of a workload (allocated
once, with torch) and runs the stages of the forward in order on one stream:

  CSA layer  ("DeepSeek-V4: Anatomy..." (modernaiengineering.com), "One query
             in a CSA layer", steps 1-5): compress the completed block(s) of
             both the KV streams and the indexer keys, score + select top-k,
             attend the selected entries, merge the sliding window.
  HCA layer  ("DeepSeek-V4 hybrid attention" (trishampatil.com) section VI):
             compress the completed block(s), attend every visible entry,
             merge the sliding window.

  Parallel    ("DeepSeek-V4 hybrid attention" (trishampatil.com) section IV: the
             attention sublayer runs the two compressed mechanisms side by side
             and concatenates their outputs): CSA and HCA on the same queries
             and window; the concatenation is the 2 n_h heads [CSA | HCA].
  SWA        (the Flash configuration's first layers, "Mastering DeepSeek-V4
             Architecture" model configurations table): the sliding window
             alone (swa_merge with no compressed branch).

Decode workloads keep the compressed caches resident (state) and write the
entry of the block that completes at this step into its cache slot; the
query is the last context token.  Prefill / forward workloads compress the
whole chunk and treat every position as a query.

Optional grouped output projection (same page, section V.3): proj = dict(w=...)
for a single attention output ([g][d_g][(n_h/g)*c] bf16, applied to `out`; a
hybrid step also takes w_h for `out_h`), or, for the parallel step, one matrix set
over the 2 n_h concatenated heads, whose first g/2 groups read the CSA heads and
the rest the HCA heads: the two halves of each projected row are written by one
grouped call each, so the concatenation is never copied.
"""
from __future__ import annotations

import torch

from . import ops
from . import workloads
from .workloads import Workload


class HybridStep:
    proj = None  # the optional grouped output projection's matrices

    def __init__(self, w: Workload, inputs: dict, fuse_window: bool = True, proj: dict | None = None):
        """fuse_window: the sliding-window merge rides on the attention call (csa_attend /
        hca_attend with a window: one launch where the whole launch fits the GPU at once;
        `out` and `lse` then hold the merged result and `o` is not written); False runs
        swa_merge as its own call after the attention."""
        self.w = w
        self.fuse_window = fuse_window
        self.x = inputs
        dev = inputs["q" if "q" in inputs else "q_h"].device
        self.device = dev
        B, c, n_h = w.batch, w.c, w.n_h
        n_q = w.n_q
        self.buf = {}
        kinds_csa = w.kind in ("forward", "csa_prefill", "csa_decode", "hybrid_decode", "parallel_decode")
        kinds_hca = w.kind in ("forward", "hca_decode", "hybrid_decode", "parallel_decode")
        self.has_csa, self.has_hca = kinds_csa, kinds_hca
        self.swa_only = w.kind == "swa_decode"
        if self.swa_only:
            self.buf["out"] = torch.empty((B, n_q, n_h, c), dtype=w.dtype, device=dev)
        f32 = torch.float32
        if kinds_csa:
            if not w.decode:
                N = w.n_csa
                self.buf["entries"] = torch.empty((B, N, c), dtype=w.dtype, device=dev)
                kI, kIs = workloads.index_key_buffers(w, B, N, dev)
                self.buf["kI"] = kI
                if kIs is not None:
                    self.buf["kI_scale"] = kIs
            self.buf["idx"] = torch.empty((B, n_q, w.k), dtype=torch.int32, device=dev)
            self.buf["o"] = torch.empty((B, n_q, n_h, c), dtype=f32, device=dev)
            self.buf["lse"] = torch.empty((B, n_q, n_h), dtype=f32, device=dev)
            self.buf["out"] = torch.empty((B, n_q, n_h, c), dtype=w.dtype, device=dev)
        if kinds_hca:
            if not w.decode:
                self.buf["entries_h"] = torch.empty((B, w.n_hca, c), dtype=w.dtype, device=dev)
            self.buf["o_h"] = torch.empty((B, n_q, n_h, c), dtype=f32, device=dev)
            self.buf["lse_h"] = torch.empty((B, n_q, n_h), dtype=f32, device=dev)
            self.buf["out_h"] = torch.empty((B, n_q, n_h, c), dtype=w.dtype, device=dev)
        self.proj = proj
        if proj is not None:
            g, d_g = proj["w"].shape[:2]
            if w.kind == "parallel_decode" and (g % 2 or proj["w"].shape[2] * g != 2 * n_h * c):
                raise ValueError("the parallel step's projection spans the 2 n_h concatenated heads")
            self.buf["proj"] = torch.empty((B, n_q, g * d_g), dtype=torch.float32, device=dev)
            if "w_h" in proj:
                g_h, d_h = proj["w_h"].shape[:2]
                self.buf["proj_h"] = torch.empty((B, n_q, g_h * d_h), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.in_branch:
            if not w.decode or w.kind in ("parallel_decode", "swa_decode"):
                raise ValueError("the in-branch operations are built for CSA / HCA / hybrid decode steps")
            # the query's position: its RoPE, and that of the entries its token completes
            self._pos = torch.full((B,), w.n_ctx - 1, dtype=torch.int64, device=dev)
        self.ws = {}
        self._size_workspaces()

    # ------------------------------------------------------------ helpers
    def _csa_tensors(self):
        x, b = self.x, self.buf
        if self.w.decode:
            return x["kc"], x["kI"], x.get("kI_scale")
        return b["entries"], b["kI"], b.get("kI_scale")

    def _hca_cache(self):
        if self.w.kind in ("hybrid_decode", "parallel_decode"):
            return self.x["kc_h"]
        return self.x["kc"] if self.w.kind == "hca_decode" else self.buf["entries_h"]

    def in_branch_args(self, branch: str):
        """RMSNorm + partial RoPE calls of a branch ("csa" or "hca"): its queries and the entry
        this step completed, both at the query's position (the block's entry takes the
        position of its last token, which is the query's)."""
        w = self.w
        if branch == "csa":
            q, entry = self.x["q"], self._csa_tensors()[0][:, w.n_csa - 1]
        else:
            q, entry = self._hca_q_kv()[0], self._hca_cache()[:, w.n_hca - 1]
        return [ops.rmsnorm_rope_args(q, pos=self._pos, rows_per_pos=w.n_h),
                ops.rmsnorm_rope_args(entry, pos=self._pos)]

    def run_in_branch(self, stream=None, branches=("csa", "hca")):
        """The in-branch RMSNorm + RoPE of the given branches, in place, as one launch (when
        the workload has the in-branch operations)."""
        if not self.w.in_branch:
            return
        calls = []
        for br in branches:
            if (br == "csa" and self.has_csa) or (br == "hca" and self.has_hca):
                calls += self.in_branch_args(br)
        ops.rmsnorm_rope_batch(calls, stream=stream)

    def sink(self, branch: str):
        """The branch's per-head attention-sink logits (None without the in-branch operations)."""
        if not self.w.in_branch:
            return None
        return self.x["sink_h"] if branch == "hca" and self.w.kind == "hybrid_decode" else self.x["sink"]

    def _hca_q_kv(self):
        """The HCA branch's queries and window rows (its own in a hybrid step's HCA layer)."""
        if self.w.kind == "hybrid_decode":
            return self.x["q_h"], self.x["kv_h"]
        return self.x["q"], self.x["kv"]

    def _size_workspaces(self):
        w, x, b = self.w, self.x, self.buf
        if self.has_csa:
            kc, kI, kIs = self._csa_tensors()
            a = ops.index_args(x["qI"], x["w"], kI, w.m, w.k, w.q_pos0, x.get("qI_scale"), kIs, b["idx"], None)
            n = ops.csa_index_topk_workspace_size(a)
            self.ws["index"] = torch.zeros(max(n, 1), dtype=torch.uint8, device=self.device)  # (counters)
            a = ops.csa_attend_args(x["q"], kc, kc, b["idx"], w.scale, b["o"], b["lse"], window=self._win_csa())
            n = int(ops._abi.load().csa_attend_workspace_size(a))
            self.ws["csa"] = torch.zeros(max(n, 1), dtype=torch.uint8, device=self.device)  # (join counters)
        if self.has_hca:
            kc = self._hca_cache()
            q = self._hca_q_kv()[0]
            a = ops.hca_attend_args(q, kc, kc, w.m_hca, w.q_pos0, w.scale, b["o_h"], b["lse_h"],
                                    window=self._win_hca())
            n = int(ops._abi.load().hca_attend_workspace_size(a))
            self.ws["hca"] = torch.zeros(max(n, 1), dtype=torch.uint8, device=self.device)

    def _kv_pos0(self):
        return self.w.n_ctx - self.w.n_win if self.w.decode else 0

    def _win_csa(self, as_dict=False):
        if not self.fuse_window:
            return None
        d = dict(kw=self.x["kv"], kv_pos0=self._kv_pos0(), q_pos0=self.w.q_pos0, n_win=self.w.n_win, out=self.buf["out"])
        if as_dict:
            return d
        return ops.window_args(d.pop("kw"), **d)

    def _win_hca(self, as_dict=False):
        if not self.fuse_window:
            return None
        kv = self._hca_q_kv()[1]
        d = dict(kw=kv, kv_pos0=self._kv_pos0(), q_pos0=self.w.q_pos0, n_win=self.w.n_win, out=self.buf["out_h"])
        if as_dict:
            return d
        return ops.window_args(d.pop("kw"), **d)

    # ------------------------------------------------------------ stages
    def compress_calls(self):
        """Argument structs of a decode step's compressions: the CSA entry and its indexer key
        completed by the block that ends at the query, and the HCA entry (each written into
        its cache slot)."""
        w, x = self.w, self.x
        st, calls = self.dev_status, []
        if self.has_csa:
            kc, kI, kIs = self._csa_tensors()
            N = w.n_csa
            calls.append(ops.compress_args(x["ca"], x["za"], x["bias"], w.m, x["cb"], x["zb"], True, N - 2, kc, None,
                                           dev_status=st, out_row0=N - 1))
            calls.append(ops.compress_args(x["kIa"], x["zIa"], x["biasI"], w.m, x["kIb"], x["zIb"], True, N - 2, kI,
                                           kIs, dev_status=st, out_row0=N - 1))
        if self.has_hca:
            Nh = w.n_hca
            calls.append(ops.compress_args(x["ch"], x["zh"], x["bias_h"], w.m_hca, first_block=Nh - 1,
                                           out=self._hca_cache(), dev_status=st, out_row0=Nh - 1))
        return calls

    def run_compress(self, stream=None):
        """A decode step's compressions as one launch (hyb_compress_batch)."""
        calls = self.compress_calls()
        if calls:
            ops.hyb_compress_batch(calls, stream=stream)

    def run_csa(self, stream=None, compress=True, in_branch=True):
        w, x, b = self.w, self.x, self.buf
        kc, kI, kIs = self._csa_tensors()
        st = self.dev_status
        if not compress:
            pass
        elif w.decode:
            N = w.n_csa
            # the block ending at the query completes entry N-1: pass blocks N-2 and N-1
            ops.hyb_compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True,
                             first_block=N - 2, out=kc, out_row0=N - 1, dev_status=st, stream=stream)
            ops.hyb_compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True,
                             first_block=N - 2, out=kI, out_scale=kIs, out_row0=N - 1, dev_status=st, stream=stream)
        else:
            ops.hyb_compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True, out=kc,
                             dev_status=st, stream=stream)
            ops.hyb_compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True, out=kI,
                             out_scale=kIs, dev_status=st, stream=stream)
        ops.csa_index_topk(x["qI"], x["w"], kI, m=w.m, k=w.k, q_pos0=w.q_pos0, qI_scale=x.get("qI_scale"),
                           kI_scale=kIs, idx=b["idx"], workspace=self.ws["index"], dev_status=st, stream=stream)
        if in_branch:
            self.run_in_branch(stream, ("csa",))
        ops.csa_attend(x["q"], kc, kc, b["idx"], scale=w.scale, o=b["o"], lse=b["lse"], workspace=self.ws["csa"],
                       dev_status=st, stream=stream, window=self._win_csa(as_dict=True), sink=self.sink("csa"))
        if not self.fuse_window:
            ops.swa_merge(x["q"], x["kv"], x["kv"], kv_pos0=self._kv_pos0(), q_pos0=w.q_pos0, n_win=w.n_win,
                          scale=w.scale, o_in=b["o"], lse_in=b["lse"], out=b["out"], dev_status=st,
                          stream=stream)

    def run_hca(self, stream=None, compress=True, in_branch=True):
        w, x, b = self.w, self.x, self.buf
        st = self.dev_status
        kc = self._hca_cache()
        q, kv = self._hca_q_kv()
        if not compress:
            pass
        elif w.decode:
            Nh = w.n_hca
            ops.hyb_compress(x["ch"], x["zh"], x["bias_h"], w.m_hca, first_block=Nh - 1, out=kc, out_row0=Nh - 1,
                             dev_status=st, stream=stream)
        else:
            ops.hyb_compress(x["ch"], x["zh"], x["bias_h"], w.m_hca, out=kc, dev_status=st, stream=stream)
        if in_branch:
            self.run_in_branch(stream, ("hca",))
        ops.hca_attend(q, kc, kc, m=w.m_hca, q_pos0=w.q_pos0, scale=w.scale, o=b["o_h"], lse=b["lse_h"],
                       workspace=self.ws["hca"], dev_status=st, stream=stream, window=self._win_hca(as_dict=True),
                       sink=self.sink("hca"))
        if not self.fuse_window:
            ops.swa_merge(q, kv, kv, kv_pos0=self._kv_pos0(), q_pos0=w.q_pos0, n_win=w.n_win, scale=w.scale,
                          o_in=b["o_h"], lse_in=b["lse_h"], out=b["out_h"], dev_status=st, stream=stream)

    def run_swa(self, stream=None):
        """A pure sliding-window layer: the window of each query, no compressed branch."""
        w, x, b = self.w, self.x, self.buf
        ops.swa_merge(x["q"], x["kv"], x["kv"], kv_pos0=self._kv_pos0(), q_pos0=w.q_pos0, n_win=w.n_win, scale=w.scale,
                      out=b["out"], dev_status=self.dev_status, stream=stream)

    def run_proj(self, stream=None):
        """The grouped output projection of the step's attention outputs (see the module notes)."""
        if self.proj is None:
            return
        b, st, W = self.buf, self.dev_status, self.proj["w"]
        if self.w.kind == "parallel_decode":
            g, d_g = W.shape[:2]
            half = (g // 2) * d_g
            ops.grouped_out_proj(b["out"], W[: g // 2], out=b["proj"][..., :half], dev_status=st, stream=stream)
            ops.grouped_out_proj(b["out_h"], W[g // 2:], out=b["proj"][..., half:], dev_status=st, stream=stream)
            return
        ops.grouped_out_proj(b["out"], W, out=b["proj"], dev_status=st, stream=stream)
        if "w_h" in self.proj:
            ops.grouped_out_proj(b["out_h"], self.proj["w_h"], out=b["proj_h"], dev_status=st, stream=stream)

    def run(self, stream=None):
        """One step.  A decode step with both layers compresses first, its three entries in
        one launch (measured: the 1M hybrid step 102.3 us batched vs 108.4 us with three
        launches; a CSA layer alone ran slower batched, 80 vs 66.5 us for Flash, so it
        keeps its two launches)."""
        if self.swa_only:
            self.run_swa(stream)
        batched = self.w.decode and self.has_csa and self.has_hca
        if batched:
            self.run_compress(stream)
            self.run_in_branch(stream)  # both layers' queries and entries, one launch
        if self.has_csa:
            self.run_csa(stream, compress=not batched, in_branch=not batched)
        if self.has_hca:
            self.run_hca(stream, compress=not batched, in_branch=not batched)
        self.run_proj(stream)

    # ------------------------------------------------------------ e2e view
    def step_input_keys(self):
        """Inputs that arrive fresh every step (the rest is resident state: caches)."""
        keys = [k for k in self.x if k not in ("kc", "kI", "kI_scale", "kc_h", "bias", "biasI", "bias_h")]
        return keys

    def output_keys(self):
        if self.proj is not None:
            return [k for k in ("proj", "proj_h") if k in self.buf]
        return [k for k in ("out", "out_h") if k in self.buf]

    def pack_step_io(self):
        """Re-home the per-step inputs and the outputs into one contiguous device
        buffer each (256-byte aligned views, current values kept), so that a step's
        host<->device traffic is one copy each way.  Returns the two uint8 buffers
        (inputs, outputs); the stages keep reading and writing the same tensors."""

        def pack(names, src):
            place, total = [], 0
            for k in names:
                nbytes = src[k].numel() * src[k].element_size()
                place.append((k, total, nbytes))
                total = (total + nbytes + 255) // 256 * 256
            flat = torch.empty(max(total, 1), dtype=torch.uint8, device=self.device)
            for k, off, nbytes in place:
                t = src[k]
                view = flat[off:off + nbytes].view(t.dtype).view(t.shape)
                view.copy_(t)
                src[k] = view
            return flat

        return pack(self.step_input_keys(), self.x), pack(self.output_keys(), self.buf)
