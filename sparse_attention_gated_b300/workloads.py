"""Workload shapes and seeded synthetic inputs.

This module holds only sizes and random draws: none of the method's
arithmetic.  Tests, the smoke check and the benchmark use it to feed the CUDA
library and the CPU oracle the same inputs.

Shapes follow the model configurations of the pages ("Mastering DeepSeek-V4
Architecture, Course 1", model configurations table; "DeepSeek-V4: Anatomy of
an Open-Source Frontier Model", CSA/HCA settings): m = 4 with overlap for CSA,
m' = 128 for HCA, c = 512, indexer 64 heads x c_I = 128, window 128, top-k
512 (Flash) or 1,024 (Pro), 64 (Flash) or 128 (Pro) query heads.

Value recipe (every draw from a torch generator seeded with the workload's
seed): compressed / raw KV values N(0,1)/sqrt(c) (N(0,1) in the float32 tiny
workload); queries N(0,1); gating logits N(0,1); positional biases N(0,1);
indexer queries and keys N(0,1) cast to e4m3 by torch (float32 in the tiny
workload) with per-row scales U(0.5, 1.5); indexer head weights w U(0,1);
attention-sink logits N(0,1) (workloads with the in-branch operations).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    # "forward" | "csa_decode" | "hca_decode" | "csa_prefill" | "hybrid_decode" (a CSA layer and an
    # HCA layer) | "parallel_decode" (CSA and HCA side by side on the same queries and window, their
    # outputs concatenated) | "swa_decode" (a pure sliding-window layer)
    kind: str
    batch: int
    n_ctx: int  # decode: tokens in context (the query is the last one); prefill/forward: chunk length
    n_h: int
    c: int
    m: int = 4
    k: int = 0
    n_ih: int = 0
    c_I: int = 0
    m_hca: int = 128
    n_win: int = 128
    dtype: torch.dtype = torch.bfloat16
    seed: int = 0
    # value scales: None = the recipe (cache / raw rows N(0,1)/sqrt(c), N(0,1) in float32);
    # parity cases also draw unit-scale rows and larger queries so that outputs are O(1)
    kv_std: float | None = None
    q_std: float = 1.0
    # grouped output projection: g groups of n_h/g heads, each mapped to d_g features
    # (16 / 1024 in the Pro configuration, 8 / 1024 in Flash)
    out_groups: int = 16
    out_dim: int = 1024
    # indexer query/key format: "e4m3" (one float32 scale per row) or "mxfp4" (e2m1 pairs,
    # one e8m0 scale per 32 dims)
    idx_fmt: str = "e4m3"
    # the in-branch operations in the step: RMSNorm + partial RoPE of the queries and of the
    # entries the step completes, and a per-head attention sink on each branch's result
    in_branch: bool = False

    @property
    def n_csa(self) -> int:
        return self.n_ctx // self.m

    @property
    def n_hca(self) -> int:
        return self.n_ctx // self.m_hca

    @property
    def idx_dtype(self) -> torch.dtype:
        if self.dtype == torch.float32:
            return torch.float32
        return torch.float4_e2m1fn_x2 if self.idx_fmt == "mxfp4" else torch.float8_e4m3fn

    @property
    def decode(self) -> bool:
        return self.kind.endswith("decode")

    @property
    def n_q(self) -> int:
        return 1 if self.decode else self.n_ctx

    @property
    def q_pos0(self) -> int:
        return self.n_ctx - 1 if self.decode else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.c)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "forward", batch=1, n_ctx=256, n_h=4, c=64, m=4, k=16, n_ih=4, c_I=32, m_hca=16,
                         n_win=16, dtype=torch.float32, seed=1001),
    "flash_csa_decode": Workload("flash_csa_decode", "csa_decode", batch=8, n_ctx=65536, n_h=64, c=512, m=4, k=512,
                                 n_ih=64, c_I=128, seed=1002, out_groups=8),
    "flash_hca_decode": Workload("flash_hca_decode", "hca_decode", batch=8, n_ctx=262144, n_h=64, c=512, m_hca=128,
                                 seed=1003, out_groups=8),
    "pro_csa_prefill": Workload("pro_csa_prefill", "csa_prefill", batch=1, n_ctx=32768, n_h=128, c=512, m=4, k=1024,
                                n_ih=64, c_I=128, seed=1004),
    "pro_1m_hybrid_decode": Workload("pro_1m_hybrid_decode", "hybrid_decode", batch=4, n_ctx=1048576, n_h=128, c=512,
                                     m=4, k=1024, n_ih=64, c_I=128, m_hca=128, seed=1005),
    # the same caches with the two branches side by side in one sublayer
    "pro_1m_parallel_decode": Workload("pro_1m_parallel_decode", "parallel_decode", batch=4, n_ctx=1048576, n_h=128,
                                       c=512, m=4, k=1024, n_ih=64, c_I=128, m_hca=128, seed=1006),
    # Flash's first layers: sliding window only
    "flash_swa_decode": Workload("flash_swa_decode", "swa_decode", batch=8, n_ctx=65536, n_h=64, c=512, seed=1007, out_groups=8),
    # the 1M decode with the in-branch operations (RMSNorm + partial RoPE, attention sinks)
    "pro_1m_hybrid_decode_in_branch": Workload("pro_1m_hybrid_decode_in_branch", "hybrid_decode", batch=4,
                                               n_ctx=1048576, n_h=128, c=512, m=4, k=1024, n_ih=64, c_I=128,
                                               m_hca=128, seed=1009, in_branch=True),
    # the 1M decode with the indexer's queries and keys in MXFP4
    "pro_1m_hybrid_decode_fp4": Workload("pro_1m_hybrid_decode_fp4", "hybrid_decode", batch=4, n_ctx=1048576, n_h=128,
                                         c=512, m=4, k=1024, n_ih=64, c_I=128, m_hca=128, seed=1008, idx_fmt="mxfp4"),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some sizes changed (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


class _Draw:
    def __init__(self, seed: int, device):
        self.device = torch.device(device)
        self.g = torch.Generator(device=self.device)
        self.g.manual_seed(seed)

    def normal(self, shape, std=1.0, dtype=torch.float32):
        x = torch.randn(shape, generator=self.g, device=self.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(dtype)

    def uniform(self, shape, lo=0.0, hi=1.0):
        x = torch.rand(shape, generator=self.g, device=self.device, dtype=torch.float32)
        return x.mul_(hi - lo).add_(lo)


def _indexer_values(d: _Draw, shape, dtype):
    """Indexer queries/keys: N(0,1), cast to e4m3 by torch, plus per-row scales U(0.5, 1.5);
    for MXFP4, uniformly random e2m1 codes (two per byte) and e8m0 block scales 2^-5 .. 2^3
    (a row's blocks within 8 binades of each other, as for rows of similar-sized values)."""
    if dtype == torch.float4_e2m1fn_x2:
        codes = torch.randint(0, 256, shape[:-1] + (shape[-1] // 2,), generator=d.g, device=d.device, dtype=torch.uint8)
        scales = torch.randint(122, 131, shape[:-1] + (shape[-1] // 32,), generator=d.g, device=d.device,
                               dtype=torch.uint8)
        return codes.view(torch.float4_e2m1fn_x2), scales.view(torch.float8_e8m0fnu)
    x = d.normal(shape)
    if dtype == torch.float32:
        return x, None
    return x.to(torch.float8_e4m3fn), d.uniform(shape[:-1], 0.5, 1.5)


def index_key_buffers(w: Workload, B: int, N: int, device):
    """Empty indexer-key buffers of N entries per sequence in w's format: (keys, scales or None)."""
    dt = w.idx_dtype
    if dt == torch.float4_e2m1fn_x2:
        return (torch.empty((B, N, w.c_I // 2), dtype=dt, device=device),
                torch.empty((B, N, w.c_I // 32), dtype=torch.float8_e8m0fnu, device=device))
    kI = torch.empty((B, N, w.c_I), dtype=dt, device=device)
    return kI, (None if dt == torch.float32 else torch.empty((B, N), dtype=torch.float32, device=device))


def make_inputs(w: Workload, device="cpu") -> dict:
    """Seeded synthetic inputs of workload w (a dict of tensors on `device`).

    Keys, by kind:
      forward / csa_prefill (every position is a query, full causal chunk):
        CSA raw rows ca, cb, za, zb [B,n,c]; bias [2m,c]; indexer raw rows
        kIa, kIb, zIa, zIb [B,n,c_I]; biasI [2m,c_I]; qI [B,n,n_ih,c_I]
        (+ qI_scale); w [B,n,n_ih]; q [B,n,n_h,c]; kv (raw window rows) [B,n,c].
        forward only: HCA raw rows ch, zh [B,n,c]; bias_h [m',c].
      csa_decode / hybrid_decode (CSA part): cache kc [B,N,c]; kI [B,N,c_I]
        (+ kI_scale); the last 2m raw rows ca, cb, za, zb [B,2m,c] and
        kIa, kIb, zIa, zIb [B,2m,c_I] (their block completes at this step);
        bias, biasI; qI, qI_scale, w, q [B,1,...]; kv [B,n_win,c] window rows.
      hca_decode / hybrid_decode (HCA part, suffix _h in hybrid): cache kc_h
        [B,N',c]; raw rows ch, zh [B,m',c]; bias_h [m',c]; q_h [B,1,n_h,c];
        kv_h [B,n_win,c].
      in-branch workloads, also: sink [n_h] float32 (sink_h for the HCA layer of a
        hybrid step).
    """
    d = _Draw(w.seed, device)
    B, n, c, dt = w.batch, w.n_ctx, w.c, w.dtype
    kv_std = w.kv_std if w.kv_std is not None else (1.0 if dt == torch.float32 else 1.0 / math.sqrt(c))
    out = {}

    def csa_raw(rows):
        out["ca"] = d.normal((B, rows, c), kv_std, dt)
        out["cb"] = d.normal((B, rows, c), kv_std, dt)
        out["za"] = d.normal((B, rows, c), 1.0, dt)
        out["zb"] = d.normal((B, rows, c), 1.0, dt)
        out["bias"] = d.normal((2 * w.m, c))
        out["kIa"] = d.normal((B, rows, w.c_I), kv_std, dt)
        out["kIb"] = d.normal((B, rows, w.c_I), kv_std, dt)
        out["zIa"] = d.normal((B, rows, w.c_I), 1.0, dt)
        out["zIb"] = d.normal((B, rows, w.c_I), 1.0, dt)
        out["biasI"] = d.normal((2 * w.m, w.c_I))

    def queries(n_q, suffix=""):
        out["q" + suffix] = d.normal((B, n_q, w.n_h, c), w.q_std, dt)

    def indexer_queries(n_q):
        qI, qs = _indexer_values(d, (B, n_q, w.n_ih, w.c_I), w.idx_dtype)
        out["qI"] = qI
        if qs is not None:
            out["qI_scale"] = qs
        out["w"] = d.uniform((B, n_q, w.n_ih))

    if w.kind in ("forward", "csa_prefill"):
        csa_raw(n)
        indexer_queries(n)
        queries(n)
        out["kv"] = d.normal((B, n, c), kv_std, dt)
        if w.kind == "forward":
            out["ch"] = d.normal((B, n, c), kv_std, dt)
            out["zh"] = d.normal((B, n, c), 1.0, dt)
            out["bias_h"] = d.normal((w.m_hca, c))
        return out

    if w.kind == "swa_decode":
        queries(1)
        out["kv"] = d.normal((B, w.n_win, c), kv_std, dt)
        return out

    if w.kind in ("csa_decode", "hybrid_decode", "parallel_decode"):
        N = w.n_csa
        out["kc"] = d.normal((B, N, c), kv_std, dt)
        kI, ks = _indexer_values(d, (B, N, w.c_I), w.idx_dtype)
        out["kI"] = kI
        if ks is not None:
            out["kI_scale"] = ks
        csa_raw(2 * w.m)
        indexer_queries(1)
        queries(1)
        out["kv"] = d.normal((B, w.n_win, c), kv_std, dt)
    if w.kind == "parallel_decode":
        # the HCA cache and its raw block; the queries and the window are the CSA branch's
        out["kc_h"] = d.normal((B, w.n_hca, c), kv_std, dt)
        out["ch"] = d.normal((B, w.m_hca, c), kv_std, dt)
        out["zh"] = d.normal((B, w.m_hca, c), 1.0, dt)
        out["bias_h"] = d.normal((w.m_hca, c))
    if w.kind in ("hca_decode", "hybrid_decode"):
        sfx = "_h" if w.kind == "hybrid_decode" else ""
        out["kc" + ("_h" if sfx else "")] = d.normal((B, w.n_hca, c), kv_std, dt)
        out["ch"] = d.normal((B, w.m_hca, c), kv_std, dt)
        out["zh"] = d.normal((B, w.m_hca, c), 1.0, dt)
        out["bias_h"] = d.normal((w.m_hca, c))
        queries(1, "_h" if sfx else "")
        out["kv" + sfx] = d.normal((B, w.n_win, c), kv_std, dt)
    if w.in_branch:
        # per-head attention-sink logits N(0,1), one set per layer
        out["sink"] = d.normal((w.n_h,))
        if w.kind == "hybrid_decode":
            out["sink_h"] = d.normal((w.n_h,))
    return out
