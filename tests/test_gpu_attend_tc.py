"""Parity of the tensor-core attention kernel (bf16, c = 512, heads in groups
of 64) against the float64 oracle, on the cases its design makes special:
key = value aliasing (the method's shared compressed entry), split lists with
a combine, ragged last tiles, whole tiles of padding, empty lists, scores that
move the softmax reference late in the list, and the window merge.

Also the two-stage top-k plan (rows longer than the shared-memory stage),
bit-exact against the oracle's selection on integer-valued scores with ties.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BF16, assert_out_close, max_abs, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _randn(g, shape, std=1.0):
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from sparse_attention_gated_b300 import ops  # noqa: F401


def _ops():
    from sparse_attention_gated_b300 import ops

    return ops


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _csa(q, kv, vv, idx, scale):
    st = _status()
    o, lse = _ops().csa_attend(q.to(DEV), kv.to(DEV), vv.to(DEV), idx.to(DEV), scale=scale, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    return to_np(o), to_np(lse)


@pytest.mark.parametrize("B,n_q,n_h,N,k,seed", [
    (4, 1, 128, 20000, 1024, 1),  # decode: 8 query-head groups, splits + combine
    (8, 1, 64, 16384, 512, 2),    # Flash decode shape
    (1, 1, 64, 3000, 300, 3),     # many splits of one group, ragged last tile
    (2, 37, 128, 900, 200, 4),    # several queries per call, one split each
])
def test_csa_attend_aliased_entries(B, n_q, n_h, N, k, seed):
    g = _gen(seed)
    c = 512
    q = _randn(g, (B, n_q, n_h, c))
    kc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(N, generator=g)[:k]).values for _ in range(n_q)])
                       for _ in range(B)]).int()
    scale = 1 / math.sqrt(c)
    o, lse = _csa(q, kc, kc, idx, scale)
    ro, rl = oracle.csa_attend(q, kc, kc, idx, scale)
    assert_out_close(o, ro)
    assert max_abs(lse, rl) <= TOL_BF16


def test_csa_attend_padding_runs_duplicates_and_empty_lists():
    """Whole tiles of -1 (at the start, in the middle), a list that is all
    padding, and repeated entries (a multiset: each repeat counts)."""
    g = _gen(5)
    B, n_q, n_h, N, k, c = 2, 3, 64, 5000, 700, 512
    q = _randn(g, (B, n_q, n_h, c))
    kc = _randn(g, (B, N, c), 2 / math.sqrt(c))
    idx = torch.randint(0, N, (B, n_q, k), generator=g).int()
    idx[0, 0, :300] = -1          # first two tiles and more: nothing
    idx[0, 1, 128:512] = -1       # three whole tiles in the middle
    idx[1, 2, :] = -1             # empty list
    idx[1, 0, 10:20] = idx[1, 0, 5]  # repeats
    scale = 1 / math.sqrt(c)
    o, lse = _csa(q, kc, kc, idx, scale)
    ro, rl = oracle.csa_attend(q, kc, kc, idx, scale)
    assert_out_close(o, ro)
    assert max_abs(lse, rl) <= TOL_BF16
    assert np.all(o[1, 2] == 0) and np.all(np.isneginf(lse[1, 2]))


@pytest.mark.parametrize("order", ["rising", "spike", "falling"])
def test_softmax_reference_moves_late_in_the_list(order):
    """Scores that span ~60 nats and peak late (or spike mid-list) force the
    lazy softmax reference to move after output has accumulated."""
    g = _gen(6)
    B, n_q, n_h, N, c = 1, 2, 64, 1500, 512
    q = _randn(g, (B, n_q, n_h, c))
    base = torch.randn((B, N, c), generator=g) / math.sqrt(c)
    if order == "rising":
        gain = torch.linspace(0.2, 12.0, N)
    elif order == "falling":
        gain = torch.linspace(12.0, 0.2, N)
    else:
        gain = torch.full((N,), 1.0)
        gain[900:905] = 14.0
    kc = (base * gain[None, :, None]).to(torch.bfloat16)
    vc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    idx = torch.arange(N, dtype=torch.int32).expand(B, n_q, N).contiguous()
    scale = 1 / math.sqrt(c) * 8
    o, lse = _csa(q, kc, vc, idx, scale)
    ro, rl = oracle.csa_attend(q, kc, vc, idx, scale)
    assert_out_close(o, ro)
    assert np.max(np.abs(lse - rl) / np.maximum(1.0, np.abs(rl))) <= 2e-3


@pytest.mark.parametrize("B,n_q,n_h,N,m,q_pos0", [
    (4, 1, 128, 8192, 128, 8192 * 128 - 1),   # 1M-context HCA decode
    (8, 1, 64, 2048, 128, 2048 * 128 - 1),    # Flash HCA decode
    (1, 1, 64, 20000, 128, 20000 * 128 - 1),  # more tiles than SMs: splits of several tiles
    (1, 300, 64, 80, 4, 0),                   # causal prefill: empty, short and ragged lists
    (2, 1, 128, 3000, 128, 2999 * 128 + 5),    # two head groups, 24 splits of one tile, ragged last tile
    (3, 2, 128, 700, 16, 700 * 16 - 18),       # two queries with different lengths, ragged tails
])
def test_hca_attend_aliased_entries(B, n_q, n_h, N, m, q_pos0):
    g = _gen(7)
    c = 512
    q = _randn(g, (B, n_q, n_h, c))
    kc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    scale = 1 / math.sqrt(c)
    st = _status()
    o, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=q_pos0, scale=scale, dev_status=st)
    assert st.item() == 0, f"device status {st.item()}"
    ro, rl = oracle.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0, scale=scale)
    assert_out_close(to_np(o), ro)
    assert max_abs(to_np(lse), rl) <= TOL_BF16


@pytest.mark.parametrize("B,n_q,n_h,n_win,kv_pos0,n_kv,q_pos0,out_dtype", [
    (4, 1, 128, 128, 2 ** 20 - 128, 128, 2 ** 20 - 1, torch.bfloat16),  # decode window
    (1, 200, 128, 128, 0, 200, 0, torch.bfloat16),                      # prefill: windows cut by the start
    (2, 3, 64, 100, 40, 300, 250, torch.float32),                       # window not a multiple of 128
    (2, 1, 128, 128, 0, 5, 4, torch.bfloat16),   # 5-row window, output dims split over 4 CTAs
    (1, 2, 64, 128, 0, 700, 600, torch.float32),  # float32 output, output dims split over 4 CTAs
])
def test_swa_merge_aliased_window(B, n_q, n_h, n_win, kv_pos0, n_kv, q_pos0, out_dtype):
    g = _gen(8)
    c = 512
    q = _randn(g, (B, n_q, n_h, c))
    kv = _randn(g, (B, n_kv, c), 1 / math.sqrt(c))
    o_in = torch.randn((B, n_q, n_h, c), generator=g) * 0.05
    lse_in = torch.randn((B, n_q, n_h), generator=g) * 2 + 5
    lse_in[0, 0, :7] = -math.inf
    scale = 1 / math.sqrt(c)
    st = _status()
    out = _ops().swa_merge(q.to(DEV), kv.to(DEV), kv.to(DEV), kv_pos0=kv_pos0, q_pos0=q_pos0, n_win=n_win,
                           scale=scale, o_in=o_in.to(DEV), lse_in=lse_in.to(DEV), out_dtype=out_dtype, dev_status=st)
    assert st.item() == 0, f"device status {st.item()}"
    ro, _ = oracle.swa_merge(q, kv, kv, kv_pos0, q_pos0, n_win, scale, o_in.double().numpy(),
                             lse_in.double().numpy())
    assert_out_close(to_np(out), ro)


def test_attention_reads_no_row_outside_the_visible_set():
    """Future entries (beyond floor((t+1)/m)) and rows past a ragged last tile
    are NaN: the outputs must not change."""
    g = _gen(9)
    B, n_q, n_h, N, m, c = 1, 40, 64, 200, 4, 512
    q = _randn(g, (B, n_q, n_h, c))
    kc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    q_pos0 = 300  # sees 75 .. 84 entries of 200
    scale = 1 / math.sqrt(c)
    o, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=q_pos0, scale=scale)
    poisoned = kc.clone()
    poisoned[:, (q_pos0 + n_q) // m:] = float("nan")
    o2, lse2 = _ops().hca_attend(q.to(DEV), poisoned.to(DEV), poisoned.to(DEV), m=m, q_pos0=q_pos0, scale=scale)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


# ------------------------------------------------------------ two-stage top-k


@pytest.mark.parametrize("B,n_q,N,k", [
    (1, 3, 40000, 512),   # chunks of 864, a short last chunk
    (2, 2, 16390, 1024),  # just past the one-stage limit: one 6-entry last chunk
    (4, 1, 262144, 1024),  # the 1M-context decode shape
    (1, 150, 20000, 256),  # more rows than SMs: the three-kernel plan
])
def test_two_stage_topk_is_bit_exact_with_ties(B, n_q, N, k):
    """Small-integer indexer inputs give exactly representable scores with many
    ties; the selection must equal the oracle's (score desc, index asc) exactly."""
    g = _gen(10)
    n_ih, c_I, m = 4, 16, 4
    qI = torch.randint(-2, 3, (B, n_q, n_ih, c_I), generator=g).float()
    kI = torch.randint(-2, 3, (B, N, c_I), generator=g).float()
    w = torch.randint(0, 3, (B, n_q, n_ih), generator=g).float()
    q_pos0 = m * N - n_q
    idx, sc = _ops().csa_index_topk(qI.to(DEV), w.to(DEV), kI.to(DEV), m=m, k=k, q_pos0=q_pos0, want_scores=True)
    ref = oracle.index_scores(qI, w, kI, m=m, q_pos0=q_pos0)
    vis = np.array([min(oracle.visible(q_pos0 + j, m), N) for j in range(n_q)])
    want = oracle.topk(ref, np.broadcast_to(vis, (B, n_q)), k)
    got = idx.cpu().numpy()
    assert np.array_equal(got, want)
    gs = sc.cpu().numpy()
    for b in range(B):
        for j in range(n_q):
            assert np.array_equal(gs[b, j], ref[b, j, want[b, j]].astype(np.float32))


# ------------------------------------------------------- fused window merge


def _fused_case(g, B, n_q, n_h, n_kv, c=512):
    q = _randn(g, (B, n_q, n_h, c))
    kv = _randn(g, (B, n_kv, c), 1 / math.sqrt(c))
    return q, kv


@pytest.mark.parametrize("B,n_q,n_h,N,k,n_win,q_pos0,n_kv,out_dtype", [
    (4, 1, 128, 20000, 1024, 128, 80000 - 1, 128, torch.bfloat16),  # decode: the window is one more split
    (2, 1, 64, 3000, 512, 100, 11999, 300, torch.float32),          # window not a tile, float32 out
    (2, 1, 128, 500, 256, 128, 40, 41, torch.bfloat16),              # window cut by the sequence start
    (1, 80, 128, 4000, 256, 128, 15000, 300, torch.bfloat16),        # many queries: one split, window after the list
])
def test_csa_attend_with_fused_window(B, n_q, n_h, N, k, n_win, q_pos0, n_kv, out_dtype):
    g = _gen(11)
    c = 512
    q, kv = _fused_case(g, B, n_q, n_h, n_kv)
    kc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    idx = torch.sort(torch.randint(0, N, (B, n_q, k), generator=g), dim=-1).values.int()
    idx[0, 0, -7:] = -1  # some padding
    kv_pos0 = q_pos0 + n_q - n_kv
    scale = 1 / math.sqrt(c)
    st = _status()
    out, lse = _ops().csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, dev_status=st,
                                 window=dict(kw=kv.to(DEV), kv_pos0=kv_pos0, q_pos0=q_pos0, n_win=n_win,
                                             out_dtype=out_dtype))
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    o, l = oracle.csa_attend(q, kc, kc, idx.numpy(), scale)
    ro, rl = oracle.swa_merge(q, kv, kv, kv_pos0, q_pos0, n_win, scale, o, l)
    assert_out_close(to_np(out), ro)
    assert max_abs(to_np(lse), rl) <= TOL_BF16


@pytest.mark.parametrize("B,n_q,n_h,N,m,q_pos0,n_win,n_kv", [
    (4, 1, 128, 8192, 128, 8192 * 128 - 1, 128, 128),  # 1M-context HCA decode + window in one launch
    (2, 1, 64, 300, 16, 300 * 16 - 5, 128, 200),       # ragged list, window at the end of the buffer
    (1, 1, 128, 3, 128, 400, 128, 401),                # a few entries, window from the sequence start
])
def test_hca_attend_with_fused_window(B, n_q, n_h, N, m, q_pos0, n_win, n_kv):
    g = _gen(12)
    c = 512
    q, kv = _fused_case(g, B, n_q, n_h, n_kv)
    kc = _randn(g, (B, N, c), 1 / math.sqrt(c))
    kv_pos0 = q_pos0 + n_q - n_kv
    scale = 1 / math.sqrt(c)
    st = _status()
    out, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=q_pos0, scale=scale, dev_status=st,
                                 window=dict(kw=kv.to(DEV), kv_pos0=kv_pos0, n_win=n_win))
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    o, l = oracle.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0, scale=scale)
    ro, rl = oracle.swa_merge(q, kv, kv, kv_pos0, q_pos0, n_win, scale, o, l)
    assert_out_close(to_np(out), ro)
    assert max_abs(to_np(lse), rl) <= TOL_BF16


def test_join_counters_reset_across_calls_of_different_shapes():
    """The splits' join counters live at the start of the workspace and every call
    leaves them zero: one zero-filled workspace serves consecutive calls of different
    shapes and split counts (and a standalone window merge in between)."""
    g = _gen(13)
    c = 512
    scale = 1 / math.sqrt(c)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    q1 = _randn(g, (4, 1, 128, c))
    kc1 = _randn(g, (4, 3000, c), 1 / math.sqrt(c))
    idx1 = torch.sort(torch.randint(0, 3000, (4, 1, 512), generator=g), dim=-1).values.int()
    q2 = _randn(g, (2, 1, 64, c))
    kc2 = _randn(g, (2, 4000, c), 1 / math.sqrt(c))
    kv2 = _randn(g, (2, 128, c), 1 / math.sqrt(c))
    ro1, rl1 = oracle.csa_attend(q1, kc1, kc1, idx1.numpy(), scale)
    o2, l2 = oracle.hca_attend(q2, kc2, kc2, m=16, q_pos0=4000 * 16 - 1, scale=scale)
    ro2, rl2 = oracle.swa_merge(q2, kv2, kv2, 4000 * 16 - 128, 4000 * 16 - 1, 128, scale, o2, l2)
    st = _status()
    for _ in range(3):
        o, lse = _ops().csa_attend(q1.to(DEV), kc1.to(DEV), kc1.to(DEV), idx1.to(DEV), scale=scale, workspace=ws,
                                   dev_status=st)
        out, lse2 = _ops().hca_attend(q2.to(DEV), kc2.to(DEV), kc2.to(DEV), m=16, q_pos0=4000 * 16 - 1, scale=scale,
                                      workspace=ws, dev_status=st,
                                      window=dict(kw=kv2.to(DEV), kv_pos0=4000 * 16 - 128, n_win=128))
        _ops().swa_merge(q2.to(DEV), kv2.to(DEV), kv2.to(DEV), kv_pos0=4000 * 16 - 128, q_pos0=4000 * 16 - 1,
                         n_win=128, scale=scale, workspace=ws[4096:], dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"device status {st.item()}"
        assert_out_close(to_np(o), ro1)
        assert max_abs(to_np(lse), rl1) <= TOL_BF16
        assert_out_close(to_np(out), ro2)
        assert max_abs(to_np(lse2), rl2) <= TOL_BF16
    assert int(ws[:1024].count_nonzero()) == 0


# ---------------------------------------------------------------- 128 heads per CTA
# Decode-shaped launches with 128 heads and key = value run the kernel that keeps all 128
# heads of a query in one CTA (each CTA one half of the output dims).  Its own cases: the
# lazy softmax reference moving mid-list (O rescaled in tensor memory), gathered lists with
# padding runs, repeats and empty lists, splits with fewer tiles than splits, a ragged last
# tile read by gather, and a fused window shorter than a tile.


@pytest.mark.parametrize("order", ["rising", "spike", "falling"])
@pytest.mark.parametrize("mode", ["csa", "hca"])
def test_h128_softmax_reference_moves_late(order, mode):
    g = _gen(16)
    B, n_h, N, c = 2, 128, 1500, 512
    q = _randn(g, (B, 1, n_h, c))
    base = torch.randn((B, N, c), generator=g) / math.sqrt(c)
    if order == "rising":
        gain = torch.linspace(0.2, 12.0, N)
    elif order == "falling":
        gain = torch.linspace(12.0, 0.2, N)
    else:
        gain = torch.full((N,), 1.0)
        gain[900:905] = 14.0
    kc = (base * gain[None, :, None]).to(torch.bfloat16)
    scale = 1 / math.sqrt(c) * 8
    st = _status()
    if mode == "csa":
        idx = torch.arange(N, dtype=torch.int32).expand(B, 1, N).contiguous()
        o, lse = _ops().csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, dev_status=st)
        ro, rl = oracle.csa_attend(q, kc, kc, idx, scale)
    else:
        o, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=4, q_pos0=4 * N - 1, scale=scale,
                                   dev_status=st)
        ro, rl = oracle.hca_attend(q, kc, kc, m=4, q_pos0=4 * N - 1, scale=scale)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_out_close(to_np(o), ro)
    assert np.max(np.abs(to_np(lse) - rl) / np.maximum(1.0, np.abs(rl))) <= 2e-3


def test_h128_csa_padding_runs_duplicates_and_empty_lists():
    g = _gen(17)
    B, n_h, N, k, c = 3, 128, 5000, 700, 512
    q = _randn(g, (B, 1, n_h, c))
    kc = _randn(g, (B, N, c), 2 / math.sqrt(c))
    idx = torch.randint(0, N, (B, 1, k), generator=g).int()
    idx[0, 0, :300] = -1          # the first tiles and more: nothing
    idx[1, 0, 128:512] = -1       # whole tiles in the middle
    idx[1, 0, 10:20] = idx[1, 0, 5]  # repeats
    idx[2, 0, :] = -1             # empty list
    scale = 1 / math.sqrt(c)
    o, lse = _csa(q, kc, kc, idx, scale)
    ro, rl = oracle.csa_attend(q, kc, kc, idx, scale)
    assert_out_close(o, ro)
    assert max_abs(lse, rl) <= TOL_BF16
    assert np.all(o[2, 0] == 0) and np.all(np.isneginf(lse[2, 0]))


@pytest.mark.parametrize("N,q_pos0,m", [
    (100, 4 * 70 - 1, 4),    # 70 visible: two tiles, the second ragged (gathered), many empty splits
    (100, 2, 4),             # nothing visible
    (64, 4 * 64 - 1, 4),     # exactly one whole tile
    (9000, 9000 * 4 - 1, 4), # long list: several tiles per split
])
def test_h128_hca_split_edges(N, q_pos0, m):
    g = _gen(18)
    B, n_h, c = 2, 128, 512
    q = _randn(g, (B, 1, n_h, c))
    kc = _randn(g, (B, N, c))  # unit-scale rows: outputs of order 0.1
    vis = min(N, (q_pos0 + 1) // m)
    kc[:, vis:] = float("nan")  # rows that must not be read
    scale = 1 / math.sqrt(c)
    st = _status()
    o, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=q_pos0, scale=scale, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ro, rl = oracle.hca_attend(q, kc[:, :max(vis, 1)], kc[:, :max(vis, 1)], m=m, q_pos0=q_pos0, scale=scale)
    if vis == 0:
        assert np.all(to_np(o) == 0) and np.all(np.isneginf(to_np(lse)))
    else:
        assert_out_close(to_np(o), ro)
        assert max_abs(to_np(lse), rl) <= TOL_BF16


@pytest.mark.parametrize("q_pos0,n_win", [(30, 128), (5000, 100), (200, 128)])
def test_h128_fused_window_shorter_than_a_tile_or_ragged(q_pos0, n_win):
    g = _gen(19)
    B, n_h, N, m, c = 2, 128, 2000, 4, 512
    q = _randn(g, (B, 1, n_h, c), 2.0)
    kc = _randn(g, (B, N, c))
    n_kv = q_pos0 + 1
    kw = _randn(g, (B, n_kv, c))
    scale = 1 / math.sqrt(c)
    st = _status()
    out, lu = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=q_pos0, scale=scale, dev_status=st,
                                window=dict(kw=kw.to(DEV), kv_pos0=0, n_win=n_win))
    torch.cuda.synchronize()
    assert st.item() == 0
    ro, rl = oracle.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0, scale=scale)
    rw, rwl = oracle.swa_merge(q, kw, kw, 0, q_pos0, n_win, scale, ro, rl)
    assert_out_close(to_np(out), rw)
    assert max_abs(to_np(lu), rwl) <= TOL_BF16


# Launches with many queries (prefill): one CTA per (query, head group, half) over its whole
# list, the window's tiles after the list's in the same softmax, no join.


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("window", [True, False])
def test_h128_many_queries_csa_lists_and_window(out_dtype, window):
    g = _gen(20)
    B, n_q, n_h, N, k, c, n_win = 2, 40, 128, 3000, 300, 512, 128
    q0 = 50  # the first queries' windows are cut by the sequence start
    q = _randn(g, (B, n_q, n_h, c), 2.0)
    kc = _randn(g, (B, N, c))
    kv = _randn(g, (B, q0 + n_q, c))
    idx = torch.sort(torch.randint(0, N, (B, n_q, k), generator=g), dim=-1).values.int()
    idx[0, 3, -100:] = -1   # ragged list ends
    idx[1, 7, :] = -1       # an empty list
    idx[1, 9, 64:192] = -1  # whole tiles of padding
    scale = 1 / math.sqrt(c)
    st = _status()
    o_ref, l_ref = oracle.csa_attend(q, kc, kc, idx.numpy(), scale)
    if window:
        out, lse = _ops().csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, dev_status=st,
                                     window=dict(kw=kv.to(DEV), kv_pos0=0, q_pos0=q0, n_win=n_win,
                                                 out_dtype=out_dtype))
        o_ref, l_ref = oracle.swa_merge(q, kv, kv, 0, q0, n_win, scale, o_ref, l_ref)
    else:
        out, lse = _ops().csa_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), idx.to(DEV), scale=scale, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    assert_out_close(to_np(out), o_ref)
    assert max_abs(to_np(lse), l_ref) <= TOL_BF16
    if not window:
        assert np.all(to_np(out)[1, 7] == 0) and np.all(np.isneginf(to_np(lse)[1, 7]))


@pytest.mark.parametrize("m,n_win", [(4, 128), (16, 100)])
def test_h128_many_queries_hca_prefill_chunk(m, n_win):
    """A prefill chunk from position 0: every query sees its own number of entries (none for
    the first m - 1, ragged last tiles) and a window cut by the chunk start."""
    g = _gen(21)
    B, n_q, n_h, c = 1, 300, 128, 512
    N = n_q // m
    q = _randn(g, (B, n_q, n_h, c), 2.0)
    kc = _randn(g, (B, N, c))
    kv = _randn(g, (B, n_q, c))
    scale = 1 / math.sqrt(c)
    st = _status()
    out, lse = _ops().hca_attend(q.to(DEV), kc.to(DEV), kc.to(DEV), m=m, q_pos0=0, scale=scale, dev_status=st,
                                 window=dict(kw=kv.to(DEV), kv_pos0=0, n_win=n_win))
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item()}"
    o, l = oracle.hca_attend(q, kc, kc, m=m, q_pos0=0, scale=scale)
    ro, rl = oracle.swa_merge(q, kv, kv, 0, 0, n_win, scale, o, l)
    assert_out_close(to_np(out), ro)
    assert max_abs(to_np(lse), rl) <= TOL_BF16
