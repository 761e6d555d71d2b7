"""The allocation-free indexer entry point (csa_index_topk_noalloc) against the
ordinary one (csa_index_topk, workspace from torch), through the C ABI.

It is meant for callers that cannot allocate device memory where they run the
indexer; its scratch is a fixed array inside the library that every call
reuses.  Two calls in a row, with different inputs, must each give exactly what
the ordinary entry point gives for the same inputs: the second call must not
see anything the first one left in the shared scratch.  The shapes take the
long-row top-k plan (threshold histograms that each call must clear).

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(seed, B, N, n_ih=64, c_I=128):
    g = torch.Generator()
    g.manual_seed(seed)
    qI = torch.randn((B, 1, n_ih, c_I), generator=g).to(torch.float8_e4m3fn)
    kI = torch.randn((B, N, c_I), generator=g).to(torch.float8_e4m3fn)
    qs = torch.rand((B, 1, n_ih), generator=g) + 0.5
    ks = torch.rand((B, N), generator=g) + 0.5
    w = torch.rand((B, 1, n_ih), generator=g)
    return [t.to(DEV) for t in (qI, kI, qs, ks, w)]


def _args(qI, kI, qs, ks, w, m, k, q_pos0, idx, scores):
    from sparse_attention_gated_b300 import ops

    return ops.index_args(qI, w, kI, m, k, q_pos0, qs, ks, idx, scores)


def _ordinary(qI, kI, qs, ks, w, m, k, q_pos0):
    from sparse_attention_gated_b300 import ops

    return ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0, qI_scale=qs, kI_scale=ks, want_scores=True)


def _noalloc(qI, kI, qs, ks, w, m, k, q_pos0):
    from sparse_attention_gated_b300 import _abi

    B = qI.shape[0]
    idx = torch.full((B, 1, k), -7, dtype=torch.int32, device=DEV)
    scores = torch.full((B, 1, k), float("nan"), dtype=torch.float32, device=DEV)
    a = _args(qI, kI, qs, ks, w, m, k, q_pos0, idx, scores)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _abi.check(_abi.load().csa_index_topk_noalloc(ctypes.byref(a), stream), "csa_index_topk_noalloc")
    return idx, scores


def test_noalloc_indexer_matches_the_ordinary_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    m, k = 4, 512
    cases = [(_inputs(61, 2, 20000), 20000), (_inputs(62, 3, 17000), 17000)]
    for inputs, N in cases:
        q_pos0 = m * N - 1  # a decode query that sees every entry
        want_idx, want_sc = _ordinary(*inputs, m, k, q_pos0)
        got_idx, got_sc = _noalloc(*inputs, m, k, q_pos0)
        torch.cuda.synchronize()
        assert torch.equal(got_idx, want_idx)
        assert torch.equal(got_sc, want_sc)
        assert (got_idx >= 0).all() and (got_idx < N).all()


def test_noalloc_indexer_recovers_after_a_timeout_through_its_reset():
    """A call whose cross-CTA waits ran out (made to, by a zero wait limit) leaves the
    counters in the library's scratch non-zero; csa_index_topk_noalloc_reset clears
    them, after which the entry point again matches the ordinary one exactly."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from sparse_attention_gated_b300 import _abi, ops

    lib = _abi.load()
    g = torch.Generator()
    g.manual_seed(63)
    m, k, B, N = 4, 512, 2, 60000
    qI = torch.randn((B, 1, 8, 64), generator=g).to(DEV)
    kI = torch.randn((B, N, 64), generator=g).to(DEV)
    w = torch.rand((B, 1, 8), generator=g).to(DEV)
    q_pos0 = m * N - 1
    want = ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        idx = torch.full((B, 1, k), -7, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        a = ops.index_args(qI, w, kI, m, k, q_pos0, idx=idx, dev_status=st)
        _abi.check(lib.csa_index_topk_noalloc(ctypes.byref(a), stream), "csa_index_topk_noalloc")
        torch.cuda.synchronize()
        return idx, st.item()

    prev = int(lib.hyb_set_grid_wait_limit(0))
    try:
        _, status = call()
    finally:
        lib.hyb_set_grid_wait_limit(prev)
    assert status & 0x2, f"status {status:#x}"
    _abi.check(lib.csa_index_topk_noalloc_reset(stream), "csa_index_topk_noalloc_reset")
    for _ in range(2):
        got, status = call()
        assert status == 0
        assert torch.equal(got, want)
