"""The parity checks themselves must be able to fail (CPU, no GPU).

With the method's input recipe (cache rows N(0,1)/sqrt(c)) an attention output
is ~1e-3 in magnitude, far below the 2e-2 absolute bar, so the output checks
also bound the error by 1% of the reference's largest magnitude.  Here the
reference is the oracle's; plausible V-path mistakes are planted in a copy of
it (an output that is zero, a split whose entries never reach the output, a
head group left out, one NaN), and the check must reject each, while the
reference rounded to bf16 (what the kernels store) passes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, max_abs, out_close


def _case(N=2048, n_h=128, c=512, m=128, seed=3):
    g = torch.Generator()
    g.manual_seed(seed)
    q = torch.randn((1, 1, n_h, c), generator=g).to(torch.bfloat16)
    kc = (torch.randn((1, N, c), generator=g) / math.sqrt(c)).to(torch.bfloat16)
    return q, kc, m, N * m - 1, 1 / math.sqrt(c)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def test_reference_rounded_to_bf16_passes():
    q, kc, m, t, scale = _case()
    ro, _ = oracle.hca_attend(q, kc, kc, m=m, q_pos0=t, scale=scale)
    assert np.abs(ro).max() < TOL_BF16  # outputs far below the absolute bar: it alone cannot fail
    assert out_close(_bf16(ro), ro)


def test_planted_v_path_mistakes_fail():
    q, kc, m, t, scale = _case()
    ro, _ = oracle.hca_attend(q, kc, kc, m=m, q_pos0=t, scale=scale)
    # all-zero output
    assert not out_close(np.zeros_like(ro), ro)
    # one of 16 splits of the entry list never reaches the output (its values zeroed)
    vz = kc.clone()
    vz[:, : kc.shape[1] // 16] = 0
    bad, _ = oracle.hca_attend(q, kc, vz, m=m, q_pos0=t, scale=scale)
    assert not out_close(_bf16(bad), ro)
    # the second head group (heads 64..127) left out
    hg = ro.copy()
    hg[:, :, 64:] = 0
    assert not out_close(hg, ro)
    # a single NaN
    nan = _bf16(ro)
    nan[0, 0, 5, 17] = np.nan
    assert max_abs(nan, ro) == float("inf") and not out_close(nan, ro)
    # values one row off (a shifted gather)
    shifted = torch.roll(kc, 1, dims=1)
    bad, _ = oracle.hca_attend(q, kc, shifted, m=m, q_pos0=t, scale=scale)
    assert not out_close(_bf16(bad), ro)


def test_max_abs_treats_nan_and_infinities_as_stated():
    a = np.array([1.0, -np.inf, np.nan])
    assert max_abs(a, a) == 0.0
    assert max_abs(a, np.array([1.0, -np.inf, 0.0])) == float("inf")
    assert max_abs(np.array([1.0, np.inf]), np.array([1.0, -np.inf])) == float("inf")
    with pytest.raises(AssertionError):
        max_abs(np.zeros(3), np.zeros(4))
