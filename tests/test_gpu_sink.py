"""Per-head attention sink on csa_attend / hca_attend against the oracle (GPU).

The sink ("DeepSeek-V4 hybrid attention" (trishampatil.com) section IV) is one more
logit per head in the softmax denominator with no value.  The library adds it to the
call's final result; the oracle's chain is attention, window merge, then
oracle.sink_merge.  Both the fused-window tensor-core path and plain calls (tensor
cores, bf16; CUDA cores, float32) are covered, and a sink of -inf must change nothing.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_gated_b300 import ops
from tests.helpers import TOL_BF16, TOL_F32, max_abs, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B, n_h, c, N, n_win, dtype):
    g = torch.Generator().manual_seed(seed)
    std = 1.0 if dtype == torch.float32 else 1.0 / math.sqrt(c)
    q = torch.randn(B, 1, n_h, c, generator=g).to(dtype)
    kc = (torch.randn(B, N, c, generator=g) * std).to(dtype)
    kw = (torch.randn(B, n_win, c, generator=g) * std).to(dtype)
    # sinks around the branch's own log-sum-exp, so that they change the result
    sink = torch.randn(n_h, generator=g) * 2.0 + math.log(N)
    return q, kc, kw, sink


def _close(got, ref, tol):
    err = max_abs(got, ref)
    return err <= tol and err <= 1e-2 * float(np.abs(ref).max())


@pytest.mark.parametrize("B,n_h,N,k", [(2, 64, 3000, 256), (1, 128, 700, 64)])
def test_csa_attend_with_window_and_sink(B, n_h, N, k):
    c, n_win = 512, 128
    q, kc, kw, sink = _inputs(81, B, n_h, c, N, n_win, torch.bfloat16)
    g = torch.Generator().manual_seed(82)
    idx = torch.sort(torch.randperm(N, generator=g)[:k].repeat(B, 1, 1), dim=-1).values.int()
    t = 10 * N + 5
    scale = 1.0 / math.sqrt(c)
    out, lse = ops.csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, sink=sink.to(DEV),
                              window=dict(kw=kw.to(DEV), kv_pos0=t - n_win + 1, q_pos0=t, n_win=n_win))
    torch.cuda.synchronize()
    o, l = oracle.csa_attend(q, kc, kc, idx.numpy(), scale)
    o, l = oracle.swa_merge(q, kw, kw, t - n_win + 1, t, n_win, scale, o, l)
    ref, ref_l = oracle.sink_merge(o, l, sink.double().numpy())
    assert _close(to_np(out), ref, TOL_BF16)
    assert max_abs(to_np(lse), ref_l) <= 1e-3


def test_hca_attend_with_window_and_sink():
    B, n_h, c, m, N, n_win = 2, 64, 512, 16, 400, 128
    q, kc, kw, sink = _inputs(83, B, n_h, c, N, n_win, torch.bfloat16)
    t = N * m - 1
    scale = 1.0 / math.sqrt(c)
    out, lse = ops.hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=t, scale=scale, sink=sink.to(DEV),
                              window=dict(kw=kw.to(DEV), kv_pos0=t - n_win + 1, n_win=n_win))
    torch.cuda.synchronize()
    o, l = oracle.hca_attend(q, kc, kc, m=m, q_pos0=t, scale=scale)
    o, l = oracle.swa_merge(q, kw, kw, t - n_win + 1, t, n_win, scale, o, l)
    ref, ref_l = oracle.sink_merge(o, l, sink.double().numpy())
    assert _close(to_np(out), ref, TOL_BF16)
    assert max_abs(to_np(lse), ref_l) <= 1e-3


@pytest.mark.parametrize("dtype,n_h,c", [(torch.bfloat16, 64, 512), (torch.float32, 4, 64)])
def test_plain_csa_attend_with_sink_then_window_merge(dtype, n_h, c):
    """Sink on (o, lse) of the compressed branch alone, then swa_merge: the same as the
    sink on the whole union (the sink's term travels in lse)."""
    B, N, k, n_win = 2, 900, 100, 16
    q, kc, kw, sink = _inputs(84, B, n_h, c, N, n_win, dtype)
    g = torch.Generator().manual_seed(85)
    idx = torch.sort(torch.randperm(N, generator=g)[:k].repeat(B, 1, 1), dim=-1).values.int()
    t = 4 * N
    scale = 1.0 / math.sqrt(c)
    o, lse = ops.csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, sink=sink.to(DEV))
    out = ops.swa_merge(q.to(DEV), kw.to(DEV), kw.to(DEV), kv_pos0=t - n_win + 1, q_pos0=t, n_win=n_win, scale=scale,
                        o_in=o, lse_in=lse, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rl = oracle.csa_attend(q, kc, kc, idx.numpy(), scale)
    so, sl = oracle.sink_merge(ro, rl, sink.double().numpy())
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert _close(to_np(o), so, tol) and max_abs(to_np(lse), sl) <= 1e-3
    ref, _ = oracle.swa_merge(q, kw, kw, t - n_win + 1, t, n_win, scale, ro, rl)
    whole, _ = oracle.sink_merge(*oracle.swa_merge(q, kw, kw, t - n_win + 1, t, n_win, scale, ro, rl),
                                 sink.double().numpy())
    assert _close(to_np(out), whole, tol)
    assert not _close(to_np(out), ref, 1e-6)  # the sink changed the result


def test_sink_of_minus_infinity_changes_nothing():
    B, n_h, c, N, k = 1, 64, 512, 500, 64
    q, kc, _, _ = _inputs(86, B, n_h, c, N, 16, torch.bfloat16)
    g = torch.Generator().manual_seed(87)
    idx = torch.sort(torch.randperm(N, generator=g)[:k].repeat(B, 1, 1), dim=-1).values.int().to(DEV)
    args = (q.to(DEV), kc.to(DEV), kc.to(DEV), idx)
    o0, l0 = ops.csa_attend(*args)
    o1, l1 = ops.csa_attend(*args, sink=torch.full((n_h,), -math.inf, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("n_q,window", [(80, False), (80, True), (1, False), (1, True)])
def test_sink_joined_by_the_128_head_kernel(n_q, window):
    """128 heads: the sink is joined where the kernel writes its final result, in one split
    per (query, half) when the queries fill the GPU (80 queries x 2 halves) and in the split
    join otherwise (one query, a long list); with and without the fused window, and a query
    with an empty list (no window: output 0, lse = the sink)."""
    B, n_h, c, N, k, n_win, q0 = 1, 128, 512, 4000, 1024, 128, 50
    g = torch.Generator().manual_seed(87)
    q = torch.randn(B, n_q, n_h, c, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, N, c, generator=g).to(torch.bfloat16)  # unit scale: outputs of order 0.1-1
    kv = torch.randn(B, q0 + n_q, c, generator=g).to(torch.bfloat16)
    sink = torch.randn(n_h, generator=g) * 2.0 + 3.0
    idx = torch.stack([torch.sort(torch.randperm(N, generator=g)[:k]).values for _ in range(n_q)])[None].int()
    if n_q > 7:
        idx[0, 7, :] = -1
    scale = 1.0 / math.sqrt(c)
    win = dict(kw=kv.to(DEV), kv_pos0=0, q_pos0=q0, n_win=n_win) if window else None
    o, lse = ops.csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, sink=sink.to(DEV),
                            window=win)
    torch.cuda.synchronize()
    ro, rl = oracle.csa_attend(q, kc, kc, idx.numpy(), scale)
    if window:
        ro, rl = oracle.swa_merge(q, kv, kv, 0, q0, n_win, scale, ro, rl)
    ref, ref_l = oracle.sink_merge(ro, rl, sink.double().numpy())
    assert _close(to_np(o), ref, TOL_BF16)
    assert max_abs(to_np(lse), ref_l) <= TOL_BF16
    if n_q > 7 and not window:
        assert np.all(to_np(o)[0, 7] == 0) and np.allclose(to_np(lse)[0, 7], sink.numpy(), atol=1e-6)
