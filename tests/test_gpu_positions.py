"""Per-query positions (a batch of sequences at different lengths): csa_index_topk,
hca_attend, swa_merge and the fused windows take an optional int64 q_pos
[B, n_q] in device memory (and kv_pos0s [B] for per-sequence window buffers).
Each batch element is checked against the oracle run at its own position,
including one before its first complete block (no entry visible), and a
position outside what exists is clipped and reported (HYB_DEV_BAD_INDEX).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, assert_out_close, check_topk_row, max_abs, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def _ops():
    from sparse_attention_gated_b300 import ops

    return ops


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("dtype,N,n_ih,c_I,k", [
    (torch.float8_e4m3fn, 20000, 64, 128, 512),  # tensor-core scores, long rows (grid top-k plan)
    (torch.float8_e4m3fn, 3000, 64, 128, 256),   # short rows (one-stage top-k)
    (torch.float32, 5000, 8, 64, 100),           # CUDA-core scores
])
def test_index_topk_with_per_query_positions(dtype, N, n_ih, c_I, k):
    g = _gen(81)
    m = 4
    pos = [m * N - 1, 1000, 2, 37]  # all entries, 250, none (before the first block), 9
    B = len(pos)
    qI = torch.randn((B, 1, n_ih, c_I), generator=g)
    kI = torch.randn((B, N, c_I), generator=g)
    w = torch.rand((B, 1, n_ih), generator=g)
    qs = ks = None
    if dtype != torch.float32:
        qI, kI = qI.to(dtype), kI.to(dtype)
        qs = torch.rand((B, 1, n_ih), generator=g) + 0.5
        ks = torch.rand((B, N), generator=g) + 0.5
    dev = lambda t: None if t is None else t.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_pos = torch.tensor(pos, dtype=torch.int64, device=DEV).view(B, 1)
    idx = _ops().csa_index_topk(dev(qI), dev(w), dev(kI), m=m, k=k, q_pos=q_pos, qI_scale=dev(qs), kI_scale=dev(ks),
                                dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    gidx = idx.cpu().numpy()
    for b, t in enumerate(pos):
        sl = slice(b, b + 1)
        s = oracle.index_scores(qI[sl], w[sl], kI[sl], m=m, q_pos0=t, qI_scale=None if qs is None else qs[sl],
                                kI_scale=None if ks is None else ks[sl])
        check_topk_row(gidx[b, 0], s[0, 0], oracle.visible(t, m), k)


def test_hca_attend_and_fused_window_with_per_sequence_positions():
    g = _gen(82)
    B, n_h, c, N, m, n_win = 4, 128, 512, 3000, 128, 128
    pos = [N * m - 1, 200000, 100, 126]  # 3000, 1562, 0 and 0 entries visible
    n_kv = 256
    kvp = [t - 130 if t >= 130 else 0 for t in pos]  # each sequence's window buffer starts elsewhere
    q = torch.randn((B, 1, n_h, c), generator=g).mul_(2).to(torch.bfloat16)
    kc = torch.randn((B, N, c), generator=g).to(torch.bfloat16)
    kw = torch.randn((B, n_kv, c), generator=g).to(torch.bfloat16)
    q_pos = torch.tensor(pos, dtype=torch.int64, device=DEV).view(B, 1)
    kv_pos0s = torch.tensor(kvp, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(c)
    ops = _ops()
    o, lse = ops.hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos=q_pos, scale=scale, dev_status=st)
    out, lu = ops.hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos=q_pos, scale=scale, dev_status=st,
                             window=dict(kw=kw.to(DEV), kv_pos0s=kv_pos0s, n_win=n_win))
    out2 = ops.swa_merge(q.to(DEV), kw.to(DEV), kw.to(DEV), q_pos=q_pos, kv_pos0s=kv_pos0s, n_win=n_win, scale=scale,
                         o_in=o, lse_in=lse, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert st.item() == 0
    for b, t in enumerate(pos):
        sl = slice(b, b + 1)
        ro, rl = oracle.hca_attend(q[sl], kc[sl], kc[sl], m=m, q_pos0=t, scale=scale)
        if oracle.visible(t, m) == 0:
            assert np.all(to_np(o[sl]) == 0) and np.all(np.isneginf(to_np(lse[sl])))
        else:
            assert_out_close(to_np(o[sl]), ro)
            assert max_abs(to_np(lse[sl]), rl) <= TOL_BF16
        rw, rwl = oracle.swa_merge(q[sl], kw[sl], kw[sl], kvp[b], t, n_win, scale, ro, rl)
        assert_out_close(to_np(out[sl]), rw)
        assert max_abs(to_np(lu[sl]), rwl) <= TOL_BF16
        assert_out_close(to_np(out2[sl]), rw)


def test_csa_attend_fused_window_with_per_sequence_positions():
    g = _gen(83)
    B, n_h, c, N, k, n_win = 3, 128, 512, 4000, 1024, 128
    pos = [40000, 700, 3]
    n_kv = 300
    kvp = [t - 200 if t >= 200 else 0 for t in pos]
    q = torch.randn((B, 1, n_h, c), generator=g).mul_(2).to(torch.bfloat16)
    kc = torch.randn((B, N, c), generator=g).to(torch.bfloat16)
    kw = torch.randn((B, n_kv, c), generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.sort(torch.randperm(N, generator=g)[:k]).values for _ in range(B)]).int().view(B, 1, k)
    idx[2, 0, :] = -1  # the sequence at position 3 has no entry yet
    q_pos = torch.tensor(pos, dtype=torch.int64, device=DEV).view(B, 1)
    kv_pos0s = torch.tensor(kvp, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(c)
    out, lu = _ops().csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, dev_status=st,
                                window=dict(kw=kw.to(DEV), q_pos=q_pos, kv_pos0s=kv_pos0s, n_win=n_win))
    torch.cuda.synchronize()
    assert st.item() == 0
    for b, t in enumerate(pos):
        sl = slice(b, b + 1)
        ro, rl = oracle.csa_attend(q[sl], kc[sl], kc[sl], idx[sl], scale)
        rw, rwl = oracle.swa_merge(q[sl], kw[sl], kw[sl], kvp[b], t, n_win, scale, ro, rl)
        assert_out_close(to_np(out[sl]), rw)
        assert max_abs(to_np(lu[sl]), rwl) <= TOL_BF16


def test_positions_outside_what_exists_are_clipped_and_reported():
    g = _gen(84)
    B, n_h, c, N, m = 2, 64, 512, 100, 128
    q = torch.randn((B, 1, n_h, c), generator=g).to(torch.bfloat16).to(DEV)
    kc = torch.randn((B, N, c), generator=g).to(torch.bfloat16).to(DEV)
    ops = _ops()
    for bad in (N * m * 3, -5):  # would see more entries than exist; negative
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        q_pos = torch.tensor([N * m - 1, bad], dtype=torch.int64, device=DEV).view(B, 1)
        o, lse = ops.hca_attend(q, kc, kc, m=m, q_pos=q_pos, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() & 0x1
        assert torch.isfinite(o).all()
    # a window row outside the buffer
    kw = torch.randn((B, 64, c), generator=g).to(torch.bfloat16).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q_pos = torch.tensor([63, 500], dtype=torch.int64, device=DEV).view(B, 1)
    out = ops.swa_merge(q, kw, kw, q_pos=q_pos, kv_pos0s=torch.zeros(B, dtype=torch.int64, device=DEV), n_win=128,
                        out_dtype=torch.float32, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & 0x1
    assert torch.isfinite(out).all()
