"""MXFP4 indexer path ("DeepSeek-V4: Anatomy of an Open-Source Frontier Model",
"FP4 quantization-aware training": V4 runs the indexer's query-key path in FP4; the
format is the OCP microscaling one, e2m1 elements in blocks of 32 with an e8m0 scale):
the compressor's MXFP4 output against the oracle's quantiser of the kernel's own float32
result (bit-exact: both sides take the rounding decisions on the same float32 values),
the indexer's scores and top-k against the oracle's scores of the decoded values, and the
1M-context decode step with MXFP4 indexer keys at full size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import check_topk_row, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def _ops():
    from sparse_attention_gated_b300 import ops

    return ops


def _unpack(t):
    """e2m1 codes (one per byte) of a float4_e2m1fn_x2 tensor: element 2i is the low nibble."""
    b = t.view(torch.uint8).cpu().numpy()
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 15
    out[..., 1::2] = b >> 4
    return out


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("c,m,overlap,B,n", [(128, 4, True, 3, 40), (512, 4, True, 2, 24), (128, 16, False, 2, 64)])
def test_compress_mxfp4_output_is_the_oracle_quantiser_of_the_float_result(c, m, overlap, B, n):
    ops = _ops()
    g = _gen(51)
    bf = torch.bfloat16
    ca, za = (torch.randn((B, n, c), generator=g).mul(0.7).to(bf).to(DEV) for _ in range(2))
    cb, zb = (torch.randn((B, n, c), generator=g).to(bf).to(DEV) for _ in range(2)) if overlap else (None, None)
    bias = torch.randn(((2 if overlap else 1) * m, c), generator=g).to(DEV)
    ref32, _ = ops.hyb_compress(ca, za, bias, m, cb=cb, zb=zb, overlap=overlap, out_dtype=torch.float32)
    q, qs = ops.hyb_compress(ca, za, bias, m, cb=cb, zb=zb, overlap=overlap, out_dtype=torch.float4_e2m1fn_x2)
    torch.cuda.synchronize()
    codes, scales = oracle.quantise_mxfp4_rows(to_np(ref32).astype(np.float32))
    assert np.array_equal(_unpack(q), codes)
    assert np.array_equal(qs.view(torch.uint8).cpu().numpy(), scales)
    # and within half a grid step of the float result
    dec = oracle.mxfp4_decode(_unpack(q), qs.view(torch.uint8).cpu().numpy())
    step = np.repeat(oracle.e8m0_decode(qs.view(torch.uint8).cpu().numpy()), 32, axis=-1)
    assert np.all(np.abs(dec - to_np(ref32)) <= 2.0 * step + 1e-12)  # (half a step; up to 2 steps where saturated)


def _fp4_case(seed, B, n_q, N, lo=120, hi=134):
    """Random codes; scale bytes in [lo, hi): a row's block exponents within 8 of each other
    for hi - lo <= 9 (the kernel folds them into the values), wider otherwise (it keeps the
    blocks apart)."""
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    r = lambda shape, a, b: torch.randint(a, b, shape, generator=g, device=DEV, dtype=torch.uint8)
    qI = r((B, n_q, 64, 64), 0, 256).view(torch.float4_e2m1fn_x2)
    qs = r((B, n_q, 64, 4), lo, hi).view(torch.float8_e8m0fnu)
    kI = r((B, N, 64), 0, 256).view(torch.float4_e2m1fn_x2)
    ks = r((B, N, 4), lo, hi).view(torch.float8_e8m0fnu)
    w = torch.rand((B, n_q, 64), generator=g, device=DEV)
    return qI, qs, kI, ks, w


def _decoded(codes_t, scales_t):
    """Decoded MXFP4 values as float32 (exact: an e2m1 value times a power of two in float32's range)."""
    return oracle.mxfp4_decode(_unpack(codes_t), scales_t.view(torch.uint8).cpu().numpy()).astype(np.float32)


@pytest.mark.parametrize("lo,hi", [(120, 134), (121, 130), (112, 121)])
@pytest.mark.parametrize("B,n_q,N,m,k,q_pos0", [
    (3, 1, 5000, 4, 512, 4 * 5000 - 1),      # decode rows: 40 tiles, the last ragged
    (2, 1, 20000, 4, 1024, 4 * 20000 - 1),   # longer rows, two runs per row
    (1, 10, 700, 4, 256, 4 * 690 - 1),       # several queries, each its own visible count
    (2, 1, 300, 4, 512, 4 * 300 - 1),        # fewer entries than k: all kept
])
def test_index_topk_mxfp4_matches_oracle(B, n_q, N, m, k, q_pos0, lo, hi):
    ops = _ops()
    qI, qs, kI, ks, w = _fp4_case(61 + N, B, n_q, N, lo, hi)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx, sc = ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=q_pos0, qI_scale=qs, kI_scale=ks, want_scores=True,
                                 dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, f"device status {st.item():#x}"
    ref = oracle.index_scores(_decoded(qI, qs), to_np(w), _decoded(kI, ks), m=m, q_pos0=q_pos0)
    gidx, gsc = to_np(idx), to_np(sc)
    for b in range(B):
        for j in range(n_q):
            vis = min(N, (q_pos0 + j + 1) // m)
            check_topk_row(gidx[b, j], ref[b, j], vis, k)
            sel = gidx[b, j][gidx[b, j] >= 0]
            # the kernel's scores of the selected entries: exact block products, float32 sums
            r_ = ref[b, j][sel]
            assert np.all(np.abs(gsc[b, j][: len(sel)] - r_) <= 1e-4 * np.maximum(np.abs(r_), 1.0))


def test_mxfp4_tiles_folded_and_blocked_in_one_row():
    """Scale spreads within 8 binades everywhere except a few key rows, which put their tiles
    on the blocked path while the neighbouring tiles stay folded, and one query head out of
    range in the second sequence, which keeps all of that query's tiles blocked."""
    ops = _ops()
    B, N, m, k = 2, 3000, 4, 256
    qI, qs, kI, ks, w = _fp4_case(71, B, 1, N, 122, 130)
    ksb = ks.view(torch.uint8)
    ksb[0, 300, 2] = 135                # tile 2 of sequence 0: one row spread 13
    ksb[0, 2047, 0] = 110               # tile 15
    qs.view(torch.uint8)[1, 0, 17, 3] = 140  # sequence 1: a head spread 18
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx, sc = ops.csa_index_topk(qI, w, kI, m=m, k=k, q_pos0=m * N - 1, qI_scale=qs, kI_scale=ks, want_scores=True,
                                 dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.index_scores(_decoded(qI, qs), to_np(w), _decoded(kI, ks), m=m, q_pos0=m * N - 1)
    for b in range(B):
        g = to_np(idx)[b, 0]
        check_topk_row(g, ref[b, 0], N, k)
        r_ = ref[b, 0][g]
        assert np.all(np.abs(to_np(sc)[b, 0] - r_) <= 1e-4 * np.maximum(np.abs(r_), 1.0))


def test_pro_1m_decode_with_mxfp4_indexer_keys_full_size():
    """The 1M-context hybrid decode step with MXFP4 indexer keys, as the benchmark runs it:
    the completed block's key compressed to MXFP4 into its cache slot, then the scores of
    all 262,144 entries and their top-1,024 for the first and last sequence."""
    from sparse_attention_gated_b300 import pipeline, workloads

    w = workloads.WORKLOADS["pro_1m_hybrid_decode_fp4"]
    x = workloads.make_inputs(w, DEV)
    step = pipeline.HybridStep(w, x)
    step.run()
    torch.cuda.synchronize()
    assert step.dev_status.item() == 0
    N = w.n_csa
    for b in (0, w.batch - 1):
        sl = slice(b, b + 1)
        cpu = lambda key: x[key][sl].cpu()
        refk = oracle.compress(cpu("kIa"), cpu("zIa"), x["biasI"].cpu(), w.m, cb=cpu("kIb"), zb=cpu("zIb"), overlap=True,
                               first_block=N - 2)[0, 0]
        dec = _decoded(x["kI"][b, N - 1:N], x["kI_scale"][b, N - 1:N])[0]
        step_sz = np.repeat(oracle.e8m0_decode(x["kI_scale"][b, N - 1].view(torch.uint8).cpu().numpy()), 32)
        assert np.all(np.abs(dec - refk) <= 2.0 * step_sz + 1e-6 * np.abs(refk).max())
        s = oracle.index_scores(_decoded(x["qI"][sl], x["qI_scale"][sl]), to_np(x["w"][sl]),
                                _decoded(x["kI"][sl], x["kI_scale"][sl]), m=w.m, q_pos0=w.n_ctx - 1)
        check_topk_row(to_np(step.buf["idx"][sl])[0, 0], s[0, 0], N, w.k)
