"""RMSNorm + partial rotary encoding (hyb_rmsnorm_rope) against the oracle (GPU).

Rows shaped like the branch's queries ([B][n_q][n_h][c], one position per query,
shared by its heads) and like compressed entries ([B][N][c], one position each),
at positions up to 2^20, in float32 and bf16."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_gated_b300 import ops
from tests.helpers import max_abs, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype,shape,rows_per_pos,rope_dims,tol", [
    (torch.float32, (2, 3, 64, 512), 64, 64, 2e-5),      # queries: heads share their query's position
    (torch.bfloat16, (2, 3, 64, 512), 64, 64, 2e-2),
    (torch.bfloat16, (4, 300, 512), 1, 64, 2e-2),         # compressed entries, one position each
    (torch.float32, (5, 7, 64), 1, 16, 2e-5),             # another width, no gain
])
def test_rmsnorm_rope_matches_the_oracle(dtype, shape, rows_per_pos, rope_dims, tol):
    g = torch.Generator().manual_seed(91)
    x = (torch.randn(*shape, generator=g) * 3.0).to(dtype)
    c = shape[-1]
    gamma = (torch.rand(c, generator=g) + 0.5) if c == 512 else None
    rows = x.numel() // c
    pos = torch.randint(0, 1 << 20, (rows // rows_per_pos,), generator=g, dtype=torch.int64)
    y = x.clone().to(DEV)
    ops.rmsnorm_rope(y, gamma=None if gamma is None else gamma.to(DEV), eps=1e-6, pos=pos.to(DEV),
                     rows_per_pos=rows_per_pos, rope_dims=rope_dims)
    torch.cuda.synchronize()
    xr = x.double().reshape(rows, c).numpy()
    ref = oracle.rmsnorm(xr, None if gamma is None else gamma.double().numpy(), eps=1e-6)
    ref = oracle.rope_partial(ref, np.repeat(pos.double().numpy(), rows_per_pos), rope_dims=rope_dims)
    got = to_np(y).reshape(rows, c)
    assert max_abs(got, ref) <= tol * max(1.0, float(np.abs(ref).max()))


def test_rmsnorm_only_without_positions():
    g = torch.Generator().manual_seed(92)
    x = torch.randn(8, 512, generator=g)
    y = ops.rmsnorm_rope(x.to(DEV), eps=0.0, pos=None)
    torch.cuda.synchronize()
    assert max_abs(to_np(y), oracle.rmsnorm(x.double().numpy(), eps=0.0)) <= 2e-5


def test_strided_rows_and_the_batched_call_match_the_oracle():
    """One cache slot of every sequence (rows N*c apart) and a query block, normalised and
    rotated as one batched launch: each against the oracle, the rows around the slot
    untouched, and bit for bit the same as the two calls made separately."""
    g = torch.Generator().manual_seed(93)
    B, N, n_h, c, slot = 4, 50, 16, 512, 37
    cache = (torch.randn(B, N, c, generator=g) * 0.05).to(torch.bfloat16).to(DEV)
    q = (torch.randn(B, 1, n_h, c, generator=g) * 2.0).to(torch.bfloat16).to(DEV)
    pos = torch.randint(0, 1 << 20, (B,), generator=g, dtype=torch.int64).to(DEV)
    cache0, q0 = cache.clone(), q.clone()
    ops.rmsnorm_rope_batch([ops.rmsnorm_rope_args(q, pos=pos, rows_per_pos=n_h),
                            ops.rmsnorm_rope_args(cache[:, slot], pos=pos)])
    c2, q2 = cache0.clone(), q0.clone()
    ops.rmsnorm_rope(q2, pos=pos, rows_per_pos=n_h)
    ops.rmsnorm_rope(c2[:, slot], pos=pos)
    torch.cuda.synchronize()
    assert torch.equal(cache, c2) and torch.equal(q, q2)
    keep = [s for s in range(N) if s != slot]
    assert torch.equal(cache[:, keep], cache0[:, keep])
    p = pos.cpu().double().numpy()
    ref_e = oracle.rope_partial(oracle.rmsnorm(to_np(cache0[:, slot])), p)
    assert max_abs(to_np(cache[:, slot]), ref_e) <= 2e-2 * max(1.0, float(np.abs(ref_e).max()))
    ref_q = oracle.rope_partial(oracle.rmsnorm(to_np(q0).reshape(B * n_h, c)), np.repeat(p, n_h))
    assert max_abs(to_np(q).reshape(B * n_h, c), ref_q) <= 2e-2 * max(1.0, float(np.abs(ref_q).max()))
