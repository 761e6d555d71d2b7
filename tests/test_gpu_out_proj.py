"""Grouped output projection ("DeepSeek-V4 hybrid attention" (trishampatil.com)
section V.3; g / d_g from the "Mastering DeepSeek-V4 Architecture" model
configurations table) on the tensor cores against the float64 oracle: group j of
n_h/g consecutive heads projected by its own d_g x (n_h/g)*c matrix, the g results
concatenated.  Decode shapes (a few rows: the weights stream once), a prefill-like
row count with a ragged last row tile, the single-group plain projection, float32
and bf16 outputs.  The oracle is run per group on the group's slice (its g = 1
case), which is what the concatenation means.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_out_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def _ops():
    from sparse_attention_gated_b300 import ops

    return ops


def _case(seed, rows, n_h, c, g, d_g):
    gen = torch.Generator()
    gen.manual_seed(seed)
    k = (n_h // g) * c
    o = torch.randn((rows, n_h, c), generator=gen).to(torch.bfloat16)
    w = (torch.randn((g, d_g, k), generator=gen) / math.sqrt(k)).to(torch.bfloat16)
    return o, w


def _reference(o, w, groups=None):
    g, d_g, _ = w.shape
    n_h = o.shape[-2]
    hg = n_h // g
    ref = {}
    for j in (range(g) if groups is None else groups):
        ref[j] = oracle.grouped_out_proj(o[..., j * hg:(j + 1) * hg, :].double().numpy(),
                                         w[j:j + 1].double().numpy())
    return ref


@pytest.mark.parametrize("rows,n_h,c,g,d_g,out_dtype,groups", [
    (4, 128, 512, 16, 1024, torch.float32, (0, 7, 15)),   # Pro decode (4 sequences)
    (8, 64, 512, 8, 1024, torch.bfloat16, (0, 3, 7)),     # Flash decode (8 sequences)
    (300, 128, 512, 16, 256, torch.bfloat16, None),        # many rows: two row tiles, the second ragged
    (1, 128, 512, 16, 128, torch.float32, None),           # a single row
])
def test_grouped_out_proj_matches_oracle(rows, n_h, c, g, d_g, out_dtype, groups):
    o, w = _case(91 + rows, rows, n_h, c, g, d_g)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _ops().grouped_out_proj(o.to(DEV), w.to(DEV), out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = to_np(out)
    # float32 outputs carry only the accumulation's rounding; bf16 outputs their own rounding too
    tol = dict(tol=1e-3, rel=1e-3) if out_dtype == torch.float32 else {}
    for j, ref in _reference(o, w, groups).items():
        assert_out_close(got[:, j * d_g:(j + 1) * d_g], ref, what=f"group {j}", **tol)


def test_grouped_out_proj_into_a_column_slice_of_a_wider_output():
    """Two grouped calls writing the two halves of each output row (the row stride of the
    output is the full width): equal to one call over the concatenated heads."""
    o, w = _case(97, 6, 64, 512, 8, 256)
    full = torch.full((6, 8 * 256), float("nan"), device=DEV)
    ops = _ops()
    ops.grouped_out_proj(o[:, :32].contiguous().to(DEV), w[:4].contiguous().to(DEV), out=full[:, :1024])
    ops.grouped_out_proj(o[:, 32:].contiguous().to(DEV), w[4:].contiguous().to(DEV), out=full[:, 1024:])
    torch.cuda.synchronize()
    ref = oracle.grouped_out_proj(o.double().numpy(), w.double().numpy())
    assert_out_close(to_np(full), ref, tol=1e-3, rel=1e-3)


def test_single_group_is_a_plain_projection_to_the_model_dimension():
    """g = 1: the concatenated features mapped by one matrix (o passed as [rows][1][K])."""
    gen = torch.Generator()
    gen.manual_seed(95)
    rows, K, d = 5, 2048, 384
    x = torch.randn((rows, 1, K), generator=gen).to(torch.bfloat16)
    w = (torch.randn((1, d, K), generator=gen) / math.sqrt(K)).to(torch.bfloat16)
    out = _ops().grouped_out_proj(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = x[:, 0].double().numpy() @ w[0].double().numpy().T
    assert_out_close(to_np(out), ref)


def test_grouped_out_proj_rejects_shapes_it_cannot_run():
    from sparse_attention_gated_b300 import _abi

    o = torch.zeros((2, 8, 512), dtype=torch.bfloat16, device=DEV)
    with pytest.raises((ValueError, _abi.HybError)):  # 3 groups do not divide 8 heads
        _ops().grouped_out_proj(o, torch.zeros((3, 128, 512 * 8 // 3), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(_abi.HybError):  # d_g not a multiple of 128
        _ops().grouped_out_proj(o, torch.zeros((2, 100, 2048), dtype=torch.bfloat16, device=DEV))
