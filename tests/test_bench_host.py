"""bench.py's host-side pieces on CPU: the oracle arm's unit of work runs for every
decode workload (scaled down to a short context), and the launch counts the benchmark
claims follow the step's composition."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from sparse_attention_gated_b300 import workloads  # noqa: E402

DECODE = [n for n, w in workloads.WORKLOADS.items() if w.decode]


@pytest.mark.parametrize("name", DECODE)
def test_oracle_arm_runs_every_decode_workload_at_a_short_context(name):
    w = workloads.WORKLOADS[name]
    w = workloads.scaled(w, n_ctx=4096, batch=1)
    x = workloads.make_inputs(w, "cpu")
    bench.oracle_query(w, x, 0)


def test_launch_counts_follow_the_step_composition():
    W = workloads.WORKLOADS
    assert bench._launches_per_step(W["pro_1m_hybrid_decode"]) == 5  # batched compression, scores, top-k, 2 attention
    assert bench._launches_per_step(W["flash_csa_decode"]) == 5  # 2 compressions, scores, top-k, attention
    assert bench._launches_per_step(W["flash_hca_decode"]) == 2
    assert bench._launches_per_step(W["flash_swa_decode"]) == 1
    # the in-branch step: one batched RMSNorm + RoPE launch; the sinks ride in the 128-head
    # attention launches, and a 64-head step adds one sink launch per layer
    assert bench._launches_per_step(W["pro_1m_hybrid_decode_in_branch"]) == 5 + 1
    flash_ib = workloads.scaled(W["flash_csa_decode"], in_branch=True)
    assert bench._launches_per_step(flash_ib) == 5 + 1 + 1
