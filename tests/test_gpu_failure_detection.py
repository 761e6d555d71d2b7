"""Failure detection without a GPU fault: the device-side waits that span CTAs
(the top-k grid plan's grid barriers, the split join of the tensor-core
attention) are bounded, and a bound that runs out must end the kernel with
HYB_DEV_TIMEOUT in dev_status, never a hang.

The tests make those waits run out on purpose by setting the library's
cross-CTA wait limit to zero cycles (hyb_set_grid_wait_limit): the first CTA
to reach a barrier then gives up at once.  Nothing faults and nothing waits
without bound: every CTA returns after its first unsatisfied check.  The call
after that one, with the default limit and its workspace counters zero-filled
again (the documented recovery), must give exactly what a clean call gives.
"""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIMEOUT = 0x2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from sparse_attention_gated_b300 import ops  # noqa: F401


def _limit(cycles):
    from sparse_attention_gated_b300 import _abi

    return int(_abi.load().hyb_set_grid_wait_limit(cycles))


def _index_inputs(seed, B, N, n_ih=8, c_I=64):
    g = torch.Generator()
    g.manual_seed(seed)
    qI = torch.randn((B, 1, n_ih, c_I), generator=g)
    kI = torch.randn((B, N, c_I), generator=g)
    w = torch.rand((B, 1, n_ih), generator=g)
    return qI.to(DEV), kI.to(DEV), w.to(DEV)


def test_topk_grid_barrier_that_runs_out_reports_a_timeout_and_the_next_call_recovers():
    from sparse_attention_gated_b300 import ops

    m, k, N = 4, 512, 60000  # two rows of 60,000 entries: the grid plan (barriers between phases)
    qI, kI, w = _index_inputs(71, 2, N)
    q_pos0 = m * N - 1
    want = ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0)
    a = ops.index_args(qI, w, kI, m, k, q_pos0, idx=torch.empty_like(want))
    ws = torch.zeros(ops.csa_index_topk_workspace_size(a), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    prev = _limit(0)
    try:
        ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        _limit(prev)
    status = st.item()
    assert status & TIMEOUT, f"status {status:#x}"
    assert 40 <= (status >> 8) & 0xFF <= 44, f"wait site {(status >> 8) & 0xFF}"
    # recovery: the counters at the workspace start are zero-filled again
    ws[: ops.csa_index_topk_counter_bytes()].zero_()
    st.zero_()
    got = ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(got, want)


def test_attention_split_join_that_runs_out_reports_a_timeout_and_the_next_call_recovers():
    from sparse_attention_gated_b300 import ops

    g = torch.Generator()
    g.manual_seed(72)
    B, n_h, N, m, c = 1, 64, 20000, 128, 512  # one query, many splits of its list
    q = torch.randn((B, 1, n_h, c), generator=g).to(torch.bfloat16).to(DEV)
    kc = (torch.randn((B, N, c), generator=g) / math.sqrt(c)).to(torch.bfloat16).to(DEV)
    q_pos0 = N * m - 1
    want_o, want_l = ops.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0)
    a = ops.hca_attend_args(q, kc, kc, m, q_pos0, 1 / math.sqrt(c), want_o, want_l)
    ws = torch.zeros(int(ops._abi.load().hca_attend_workspace_size(a)), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    prev = _limit(0)
    try:
        ops.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        _limit(prev)
    status = st.item()
    assert status & TIMEOUT, f"status {status:#x}"
    assert (status >> 8) & 0xFF == 18, f"wait site {(status >> 8) & 0xFF}"
    ws[:1024].zero_()  # the join counters
    st.zero_()
    o, lse = ops.hca_attend(q, kc, kc, m=m, q_pos0=q_pos0, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o, want_o) and torch.equal(lse, want_l)
