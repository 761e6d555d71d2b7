"""Incremental decode session against the oracle, token by token (GPU).

A prefix is ingested (caches compressed in one call, rings filled), then tokens
are decoded one at a time across CSA and HCA block boundaries and window wraps.
After every token the session's caches must equal the oracle's compression of the
whole history, its selection must be a top-k of the oracle's scores over the
session's key cache, and both layers' outputs must equal the oracle's chain (the
selected entries' attention merged with the window) over the same history.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_gated_b300.session import DecodeSession
from tests.helpers import TOL_BF16, check_topk_row, max_abs, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

B, NH, C, M, MH, K, NIH, CI, W = 2, 64, 512, 4, 16, 64, 64, 128, 32
N0, T = 301, 360  # prefix length, last position + 1


def _history(seed):
    """Seeded rows for positions 0..T-1 (the shapes and value recipe of the decode
    workloads: KV rows N(0,1)/sqrt(c), gate logits and queries N(0,1), indexer queries
    e4m3 with U(0.5, 1.5) scales, indexer weights U(0,1))."""
    g = torch.Generator().manual_seed(seed)
    kv_std = 1.0 / math.sqrt(C)
    n = lambda *s, std=1.0: (torch.randn(*s, generator=g) * std).to(torch.bfloat16)
    h = {s: n(B, T, C, std=kv_std) for s in ("ca", "cb", "ch", "kv", "kv_h")}
    h.update({s: n(B, T, C) for s in ("za", "zb", "zh")})
    h.update({s: n(B, T, CI, std=kv_std) for s in ("kIa", "kIb")})
    h.update({s: n(B, T, CI) for s in ("zIa", "zIb")})
    h["q"], h["q_h"] = n(B, T, NH, C), n(B, T, NH, C)
    h["qI"] = torch.randn(B, T, NIH, CI, generator=g).to(torch.float8_e4m3fn)
    h["qI_scale"] = torch.rand(B, T, NIH, generator=g) + 0.5
    h["w"] = torch.rand(B, T, NIH, generator=g)
    bias = torch.randn(2 * M, C, generator=g)
    biasI = torch.randn(2 * M, CI, generator=g)
    bias_h = torch.randn(MH, C, generator=g)
    return h, bias, biasI, bias_h


ROW_STREAMS = ("ca", "cb", "za", "zb", "kIa", "kIb", "zIa", "zIb", "ch", "zh", "kv", "kv_h")


def _close(got, ref):
    """The stated bf16 bound (max-abs 2e-2) and, since these values are small (KV rows
    of scale 1/sqrt(c)), also 1% of the reference's largest magnitude."""
    err = max_abs(got, ref)
    return err <= TOL_BF16 and err <= 1e-2 * float(np.abs(ref).max())


def test_decode_session_matches_the_oracle_token_by_token():
    h, bias, biasI, bias_h = _history(71)
    s = DecodeSession(batch=B, n_max=512, n_h=NH, c=C, m=M, m_hca=MH, k=K, n_ih=NIH, c_I=CI, n_win=W, bias=bias,
                      biasI=biasI, bias_h=bias_h, device=DEV)
    s.prefill({k: h[k][:, :N0].contiguous().to(DEV) for k in ROW_STREAMS})
    scale = 1.0 / math.sqrt(C)
    for t in range(N0, T):
        s.append({k: h[k][:, t].contiguous().to(DEV) for k in ROW_STREAMS})
        at = lambda k: h[k][:, t].contiguous().to(DEV)
        out, out_h = s.step(q=at("q"), qI=at("qI"), qI_scale=at("qI_scale"), w=at("w"), q_h=at("q_h"))
        torch.cuda.synchronize()
        assert s.dev_status.item() == 0, f"t={t}: device status {s.dev_status.item()}"
        assert s.t == t + 1
        nv, nvh = (t + 1) // M, (t + 1) // MH
        hist = {k: h[k][:, :t + 1] for k in ROW_STREAMS}
        # caches = the oracle's compression of the whole history
        kc = s.csa_kc[:, :nv].cpu()
        ref = oracle.compress(hist["ca"], hist["za"], bias, M, cb=hist["cb"], zb=hist["zb"], overlap=True)
        assert ref.shape[1] == nv and _close(to_np(kc), ref), f"t={t}: CSA entries"
        refI = oracle.compress(hist["kIa"], hist["zIa"], biasI, M, cb=hist["kIb"], zb=hist["zIb"], overlap=True)
        kI, kIs = s.csa_kI[:, :nv].cpu(), s.csa_kIs[:, :nv].cpu()
        dec = kI.float().numpy() * kIs.numpy()[..., None]
        amax = np.abs(refI).max(axis=-1, keepdims=True)
        assert np.all(np.abs(dec - refI) <= amax / 16 + 1e-6), f"t={t}: FP8 index keys"
        hkc = s.hca_kc[:, :nvh].cpu()
        refh = oracle.compress(hist["ch"], hist["zh"], bias_h, MH)
        assert refh.shape[1] == nvh and _close(to_np(hkc), refh), f"t={t}: HCA entries"
        # selection: a top-k of the oracle's scores over the session's key cache
        q1 = lambda x: x[:, t:t + 1]
        sc = oracle.index_scores(q1(h["qI"]), q1(h["w"]), kI, m=M, q_pos0=t, qI_scale=q1(h["qI_scale"]), kI_scale=kIs)
        idx = s.idx.cpu().numpy()
        for b in range(B):
            check_topk_row(idx[b, 0], sc[b, 0], nv, K)
        # both layers: attention of the session's entries merged with the window
        o, l = oracle.csa_attend(q1(h["q"]), kc, kc, idx, scale)
        ref_out, _ = oracle.swa_merge(q1(h["q"]), hist["kv"], hist["kv"], 0, t, W, scale, o, l)
        assert _close(to_np(out), ref_out), f"t={t}: CSA layer output"
        o, l = oracle.hca_attend(q1(h["q_h"]), hkc, hkc, m=MH, q_pos0=t, scale=scale)
        ref_out, _ = oracle.swa_merge(q1(h["q_h"]), hist["kv_h"], hist["kv_h"], 0, t, W, scale, o, l)
        assert _close(to_np(out_h), ref_out), f"t={t}: HCA layer output"


def test_decode_session_with_sequences_at_different_lengths():
    """Three sequences with prefixes of 301, 250 and 2 tokens (the last one before its
    first complete block) decode 40 tokens each: blocks complete at different steps,
    the calls take per-sequence positions, and every sequence must match the oracle
    over its own history after every token."""
    h, bias, biasI, bias_h = _history(72)
    lengths = [301, 250, 2]
    Bq = len(lengths)
    h3, _, _, _ = _history(73)  # the history has B = 2 sequences: a third from another seed
    hh = {k: torch.cat([h[k], h3[k][:1]]) for k in h}
    s = DecodeSession(batch=Bq, n_max=512, n_h=NH, c=C, m=M, m_hca=MH, k=K, n_ih=NIH, c_I=CI, n_win=W, bias=bias,
                      biasI=biasI, bias_h=bias_h, device=DEV)
    n0 = max(lengths)
    s.prefill({k: hh[k][:, :n0].contiguous().to(DEV) for k in ROW_STREAMS}, lengths=lengths)
    scale = 1.0 / math.sqrt(C)
    for step in range(40):
        tb = list(s.tb)
        rows = {k: torch.stack([hh[k][b, tb[b]] for b in range(Bq)]).to(DEV) for k in ROW_STREAMS}
        s.append(rows)
        at = lambda k: torch.stack([hh[k][b, tb[b]] for b in range(Bq)]).to(DEV)
        out, out_h = s.step(q=at("q"), qI=at("qI"), qI_scale=at("qI_scale"), w=at("w"), q_h=at("q_h"))
        torch.cuda.synchronize()
        assert s.dev_status.item() == 0, f"step {step}: device status {s.dev_status.item()}"
        assert s.tb == [t + 1 for t in tb]
        for b, t in enumerate(tb):
            sl = slice(b, b + 1)
            nv, nvh = (t + 1) // M, (t + 1) // MH
            hist = {k: hh[k][sl, :t + 1] for k in ROW_STREAMS}
            kc = s.csa_kc[sl, :nv].cpu()
            if nv:
                ref = oracle.compress(hist["ca"], hist["za"], bias, M, cb=hist["cb"], zb=hist["zb"], overlap=True)
                assert _close(to_np(kc), ref), f"step {step}, sequence {b}: CSA entries"
            kI, kIs = s.csa_kI[sl, :nv].cpu(), s.csa_kIs[sl, :nv].cpu()
            q1 = lambda x: x[sl, t:t + 1]
            if nv:
                sc = oracle.index_scores(q1(hh["qI"]), q1(hh["w"]), kI, m=M, q_pos0=t, qI_scale=q1(hh["qI_scale"]),
                                         kI_scale=kIs)
                check_topk_row(s.idx[b, 0].cpu().numpy(), sc[0, 0], nv, K)
            idx = s.idx[sl].cpu().numpy()
            o, l = oracle.csa_attend(q1(hh["q"]), kc, kc, idx, scale)
            ref_out, _ = oracle.swa_merge(q1(hh["q"]), hist["kv"], hist["kv"], 0, t, W, scale, o, l)
            assert _close(to_np(out[sl]), ref_out), f"step {step}, sequence {b}: CSA layer output"
            hkc = s.hca_kc[sl, :nvh].cpu()
            o, l = oracle.hca_attend(q1(hh["q_h"]), hkc, hkc, m=MH, q_pos0=t, scale=scale)
            ref_out, _ = oracle.swa_merge(q1(hh["q_h"]), hist["kv_h"], hist["kv_h"], 0, t, W, scale, o, l)
            assert _close(to_np(out_h[sl]), ref_out), f"step {step}, sequence {b}: HCA layer output"
