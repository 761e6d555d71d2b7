"""GPU parity: every library call against the float64 oracle, element by element.

Sizes span several tiles and ragged tails; the full-size workloads are
checked in test_gpu_fullsize.py on sampled rows.  All calls go through the
C ABI (sparse_attention_gated_b300.ops -> libhyb.so).
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, TOL_F32, assert_out_close, check_topk_row, max_abs, to_np

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_attention_gated_b300 import ops, pipeline, workloads

DEV = "cuda"


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn(g, shape, dtype=torch.float32, std=1.0):
    return (torch.randn(shape, generator=g) * std).to(dtype)


# ---------------------------------------------------------------- compress


@pytest.mark.parametrize("dtype,c,m,overlap,n,B,first_block", [
    (torch.float32, 64, 4, True, 256, 1, 0),
    (torch.float32, 64, 16, False, 256, 1, 0),
    (torch.bfloat16, 512, 4, True, 4 * 37 + 3, 2, 0),      # ragged tail
    (torch.bfloat16, 512, 128, False, 128 * 5 + 17, 2, 0),
    (torch.bfloat16, 128, 4, True, 8, 3, 9),               # decode append form
    (torch.bfloat16, 512, 128, False, 128, 4, 41),
    (torch.float32, 32, 4, True, 4 * 3, 1, 0),
])
def test_compress_matches_oracle(dtype, c, m, overlap, n, B, first_block):
    g = _gen(11)
    std = 1.0 if dtype == torch.float32 else 1 / math.sqrt(c)
    ca, cb = _randn(g, (B, n, c), dtype, std), _randn(g, (B, n, c), dtype, std)
    za, zb = _randn(g, (B, n, c), dtype), _randn(g, (B, n, c), dtype)
    bias = _randn(g, (2 * m if overlap else m, c))
    kw = dict(cb=cb.to(DEV), zb=zb.to(DEV)) if overlap else {}
    out, _ = ops.hyb_compress(ca.to(DEV), za.to(DEV), bias.to(DEV), m, overlap=overlap, first_block=first_block,
                              out_dtype=torch.float32, **kw)
    ref = oracle.compress(ca, za, bias, m, cb=cb if overlap else None, zb=zb if overlap else None, overlap=overlap,
                          first_block=first_block)
    assert out.shape == ref.shape
    got = to_np(out)
    assert max_abs(got, ref) <= 1e-5 * max(1.0, np.abs(ref).max())
    # bf16 output = the float32 result rounded to nearest even
    outb, _ = ops.hyb_compress(ca.to(DEV), za.to(DEV), bias.to(DEV), m, overlap=overlap, first_block=first_block,
                               out_dtype=torch.bfloat16, **kw)
    assert torch.equal(outb.cpu(), out.cpu().to(torch.bfloat16))


@pytest.mark.parametrize("c,B,n", [(128, 2, 4 * 50 + 2), (128, 1, 8), (64, 3, 4 * 9)])
def test_compress_fp8_output_is_the_oracle_quantiser_of_the_float_result(c, B, n):
    """E4M3 codes and scales must be bit-exact against the oracle's quantiser fed
    the kernel's own float32 entries (the decision is taken in float32 on both sides)."""
    g = _gen(12)
    std = 1 / math.sqrt(c)
    t = [_randn(g, (B, n, c), torch.bfloat16, s).to(DEV) for s in (std, std, 1.0, 1.0)]
    bias = _randn(g, (8, c)).to(DEV)
    f32, _ = ops.hyb_compress(t[0], t[2], bias, 4, cb=t[1], zb=t[3], overlap=True, out_dtype=torch.float32)
    q8, sc = ops.hyb_compress(t[0], t[2], bias, 4, cb=t[1], zb=t[3], overlap=True, out_dtype=torch.float8_e4m3fn)
    codes, scales = oracle.quantise_fp8_rows(f32.cpu().numpy())
    assert np.array_equal(q8.cpu().view(torch.uint8).numpy(), codes)
    assert np.array_equal(sc.cpu().numpy(), scales)
    # and the decoded entries stay within one e4m3 step of the float64 oracle
    ref = oracle.compress(*[x.cpu() for x in (t[0], t[2])], bias.cpu(), 4, cb=t[1].cpu(), zb=t[3].cpu(), overlap=True)
    dec = oracle.e4m3_decode(codes) * scales[..., None]
    x = np.abs(ref) / scales[..., None]  # magnitude in code units
    step_code = np.where(x >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(x, 1e-30))) - 3), 2.0 ** -9)
    assert np.all(np.abs(dec - ref) <= step_code * scales[..., None] * 1.0001)


def test_compress_batch_equals_the_separate_calls():
    """The decode step's three compressions in one launch (CSA entry with overlap, its FP8
    indexer key, HCA entry, written into cache slots) are bit-identical to three
    hyb_compress calls, and the CSA entry also matches the oracle."""
    g = _gen(31)
    B, c, cI, m, mh, N, Nh = 3, 512, 128, 4, 128, 20, 6
    bf = torch.bfloat16
    ca, cb, za, zb = (_randn(g, (B, 2 * m, c), std=0.3).to(bf) for _ in range(4))
    kIa, kIb, zIa, zIb = (_randn(g, (B, 2 * m, cI)).to(bf) for _ in range(4))
    ch, zh = (_randn(g, (B, mh, c)).to(bf) for _ in range(2))
    bias, biasI, bias_h = _randn(g, (2 * m, c)), _randn(g, (2 * m, cI)), _randn(g, (mh, c))
    d = {k: v.to(DEV) for k, v in dict(ca=ca, cb=cb, za=za, zb=zb, kIa=kIa, kIb=kIb, zIa=zIa, zIb=zIb, ch=ch, zh=zh,
                                        bias=bias, biasI=biasI, bias_h=bias_h).items()}
    outs = []
    for batched in (False, True):
        kc = torch.zeros((B, N, c), dtype=bf, device=DEV)
        kI = torch.zeros((B, N, cI), dtype=torch.float8_e4m3fn, device=DEV)
        kIs = torch.zeros((B, N), device=DEV)
        kh = torch.zeros((B, Nh, c), dtype=bf, device=DEV)
        calls = [ops.compress_args(d["ca"], d["za"], d["bias"], m, d["cb"], d["zb"], True, N - 2, kc, None,
                                   out_row0=N - 1),
                 ops.compress_args(d["kIa"], d["zIa"], d["biasI"], m, d["kIb"], d["zIb"], True, N - 2, kI, kIs,
                                   out_row0=N - 1),
                 ops.compress_args(d["ch"], d["zh"], d["bias_h"], mh, first_block=Nh - 1, out=kh, out_row0=Nh - 1)]
        if batched:
            ops.hyb_compress_batch(calls)
        else:
            lib = ops._abi.load()
            for a in calls:
                ops._abi.check(lib.hyb_compress(ctypes.byref(a), None, 0, None), "hyb_compress")
        torch.cuda.synchronize()
        outs.append((kc, kI.view(torch.uint8), kIs, kh))
    for x, y in zip(*outs):
        assert torch.equal(x, y)
    ref = oracle.compress(ca, za, bias, m, cb=cb, zb=zb, overlap=True, first_block=N - 2)
    assert max_abs(to_np(outs[1][0][:, N - 1:]), ref) <= 2.0 ** -7 * max(np.abs(ref).max(), 1e-3)


def test_compress_writes_into_a_cache_slot():
    g = _gen(13)
    B, c, m, N = 2, 512, 4, 10
    rows = [_randn(g, (B, 2 * m, c), torch.bfloat16).to(DEV) for _ in range(4)]
    bias = _randn(g, (2 * m, c)).to(DEV)
    cache = torch.zeros((B, N, c), dtype=torch.bfloat16, device=DEV)
    ops.hyb_compress(rows[0], rows[2], bias, m, cb=rows[1], zb=rows[3], overlap=True, first_block=6, out=cache,
                     out_row0=7)
    ref = oracle.compress(*[r.cpu() for r in (rows[0], rows[2])], bias.cpu(), m, cb=rows[1].cpu(), zb=rows[3].cpu(),
                          overlap=True, first_block=6)
    got = to_np(cache)
    assert np.all(got[:, :7] == 0) and np.all(got[:, 8:] == 0)
    assert max_abs(got[:, 7], ref[:, 0]) < 2 ** -7 * np.abs(ref).max() + 1e-6


# ------------------------------------------------------------ index + top-k


def _index_case(seed, B, n_q, N, n_ih, c_I, m, q_pos0, fp8):
    g = _gen(seed)
    if fp8:
        qI = _randn(g, (B, n_q, n_ih, c_I)).to(torch.float8_e4m3fn)
        kI = _randn(g, (B, N, c_I)).to(torch.float8_e4m3fn)
        qs = (torch.rand((B, n_q, n_ih), generator=g) + 0.5)
        ks = (torch.rand((B, N), generator=g) + 0.5)
    else:
        qI, kI = _randn(g, (B, n_q, n_ih, c_I)), _randn(g, (B, N, c_I))
        qs = ks = None
    w = torch.rand((B, n_q, n_ih), generator=g)
    return qI, kI, qs, ks, w


def _run_index(qI, kI, qs, ks, w, m, k, q_pos0, N):
    dev = lambda t: None if t is None else t.to(DEV)
    idx, sc = ops.csa_index_topk(dev(qI), dev(w), dev(kI), m=m, k=k, q_pos0=q_pos0, qI_scale=dev(qs),
                                 kI_scale=dev(ks), n_entries=N, want_scores=True)
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("fp8,B,n_q,N,n_ih,c_I,m,k,q_pos0", [
    (False, 1, 256, 64, 4, 32, 4, 16, 0),          # the tiny workload's shape: every position a query
    (True, 2, 40, 3000, 64, 128, 4, 512, 12000 - 40),
    (True, 2, 1, 20000, 64, 128, 4, 512, 80000 - 1),  # decode row longer than the shared-memory stage
    (True, 4, 1, 262144, 64, 128, 4, 1024, 4 * 262144 - 1),  # 1M-context decode rows
    (True, 1, 6, 700, 64, 128, 4, 1024, 2795),      # fewer visible entries than k
    (False, 3, 17, 333, 16, 64, 4, 100, 1000),
])
def test_index_topk_matches_oracle(fp8, B, n_q, N, n_ih, c_I, m, k, q_pos0):
    qI, kI, qs, ks, w = _index_case(21, B, n_q, N, n_ih, c_I, m, q_pos0, fp8)
    idx, sel_scores = _run_index(qI, kI, qs, ks, w, m, k, q_pos0, N)
    ref = oracle.index_scores(qI, w, kI, m=m, q_pos0=q_pos0, qI_scale=qs, kI_scale=ks)
    tol = 1e-5 if not fp8 else 1e-4
    kinds = []
    for b in range(B):
        for j in range(n_q):
            vis = min(oracle.visible(q_pos0 + j, m), N)
            kinds.append(check_topk_row(idx[b, j], ref[b, j], vis, k))
            take = min(k, vis)
            sel = idx[b, j, :take]
            got = sel_scores[b, j, :take]
            exp = ref[b, j, sel]
            assert np.all(np.abs(got - exp) <= tol * np.maximum(1.0, np.abs(exp))), "selected scores"
            assert np.all(np.isneginf(sel_scores[b, j, take:]))


def test_index_topk_counters_reset_across_calls_of_different_shapes():
    """One zero-filled workspace serves consecutive index + top-k calls of different
    shapes (two decode batches with different row counts and lengths, and a prefill
    block), in turn.  Every call must match the oracle and leave the workspace's
    counters zero."""
    cases = [
        (4, 1, 80000, 64, 128, 4, 512, 4 * 80000 - 1),
        (2, 1, 20000, 64, 128, 4, 512, 80000 - 1),
        (1, 40, 3000, 64, 128, 4, 256, 12000 - 40),      # prefill kernel
    ]
    inputs = [(_index_case(31 + i, B, n_q, N, n_ih, c_I, m, q_pos0, True), (B, n_q, N, m, k, q_pos0))
              for i, (B, n_q, N, n_ih, c_I, m, k, q_pos0) in enumerate(cases)]
    refs = [oracle.index_scores(qI, w, kI, m=m, q_pos0=q_pos0, qI_scale=qs, kI_scale=ks)
            for (qI, kI, qs, ks, w), (B, n_q, N, m, k, q_pos0) in inputs]
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    n_zero = ops.csa_index_topk_counter_bytes()
    assert 0 < n_zero < ws.numel()
    for _ in range(2):
        for ((qI, kI, qs, ks, w), (B, n_q, N, m, k, q_pos0)), ref in zip(inputs, refs):
            idx = ops.csa_index_topk(qI.to(DEV), w.to(DEV), kI.to(DEV), m=m, k=k, q_pos0=q_pos0,
                                     qI_scale=qs.to(DEV), kI_scale=ks.to(DEV), n_entries=N, workspace=ws,
                                     dev_status=st)
            torch.cuda.synchronize()
            assert st.item() == 0, f"device status {st.item()}"
            idx = idx.cpu().numpy()
            for b in range(B):
                for j in range(n_q):
                    check_topk_row(idx[b, j], ref[b, j], min(oracle.visible(q_pos0 + j, m), N), k)
            assert int(ws[:n_zero].count_nonzero()) == 0


def test_scoring_events_outside_a_graph():
    """The scoring-kernel events may be passed on a stream that is not being captured:
    the call records them plainly, the result is unchanged and they bracket the kernel."""
    qI, kI, qs, ks, w = _index_case(41, 2, 1, 20000, 64, 128, 4, 80000 - 1, True)
    args = [t.to(DEV) for t in (qI, w, kI)]
    kw = dict(m=4, k=512, q_pos0=80000 - 1, qI_scale=qs.to(DEV), kI_scale=ks.to(DEV), n_entries=20000)
    plain = ops.csa_index_topk(*args, **kw)
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in ev:
        e.record()  # torch only times events it has seen recorded; the library records them again
    timed = ops.csa_index_topk(*args, **kw, scores_events=ev)
    torch.cuda.synchronize()
    assert torch.equal(plain, timed)
    assert ev[0].elapsed_time(ev[1]) > 0


def test_topk_is_bit_exact_with_integer_scores_and_ties():
    """Small-integer indexer inputs make every score exact in float32, so the
    selection (including the lower-index tie rule) must equal the oracle's exactly."""
    g = _gen(22)
    B, n_q, N, n_ih, c_I, m, k = 2, 64, 3000, 4, 16, 4, 100
    qI = torch.randint(-2, 3, (B, n_q, n_ih, c_I), generator=g).float()
    kI = torch.randint(-2, 3, (B, N, c_I), generator=g).float()
    w = torch.randint(0, 3, (B, n_q, n_ih), generator=g).float()
    q_pos0 = 4 * N - n_q
    idx, _ = _run_index(qI, kI, None, None, w, m, k, q_pos0, N)
    ref = oracle.index_scores(qI, w, kI, m=m, q_pos0=q_pos0)
    vis = [min(oracle.visible(q_pos0 + j, m), N) for j in range(n_q)]
    want = oracle.topk(ref, np.broadcast_to(np.array(vis), (B, n_q)), k)
    assert np.array_equal(idx, want)


# ---------------------------------------------------------------- attention


def _attn_inputs(seed, B, n_q, n_h, c, N, dtype, distinct_v=True):
    g = _gen(seed)
    std = 1.0 if dtype == torch.float32 else 1 / math.sqrt(c)
    q = _randn(g, (B, n_q, n_h, c), dtype)
    kc = _randn(g, (B, N, c), dtype, std * 4)
    vc = _randn(g, (B, N, c), dtype, std) if distinct_v else kc
    return q, kc, vc


@pytest.mark.parametrize("dtype,B,n_q,n_h,c,N,k", [
    (torch.float32, 1, 64, 4, 64, 64, 16),
    (torch.bfloat16, 2, 3, 64, 512, 5000, 512),      # long lists: split-KV path
    (torch.bfloat16, 1, 9, 128, 512, 2048, 1024),
    (torch.float32, 2, 5, 8, 128, 300, 37),
])
def test_csa_attend_matches_oracle(dtype, B, n_q, n_h, c, N, k):
    q, kc, vc = _attn_inputs(31, B, n_q, n_h, c, N, dtype)
    g = _gen(32)
    idx = torch.stack([torch.stack([torch.sort(torch.randperm(N, generator=g)[:k]).values for _ in range(n_q)])
                       for _ in range(B)]).int()
    idx[0, 0, k // 2:] = -1  # padded row
    if n_q > 1:
        idx[-1, 1, :] = -1    # empty row
    scale = 1 / math.sqrt(c)
    o, lse = ops.csa_attend(q.to(DEV), kc.to(DEV), vc.to(DEV), idx.to(DEV), scale=scale)
    ro, rl = oracle.csa_attend(q, kc, vc, idx, scale)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_out_close(to_np(o), ro, tol)
    assert max_abs(to_np(lse), rl) <= tol
    if n_q > 1:
        assert np.all(to_np(o)[-1, 1] == 0) and np.all(np.isneginf(to_np(lse)[-1, 1]))


@pytest.mark.parametrize("dtype,B,n_q,n_h,c,N,m,q_pos0", [
    (torch.float32, 1, 256, 4, 64, 16, 16, 0),          # tiny workload: includes queries with no entry
    (torch.bfloat16, 2, 1, 64, 512, 2048, 128, 262143),  # decode: split-KV
    (torch.bfloat16, 1, 4, 128, 512, 700, 128, 128 * 700 - 4),
    (torch.float32, 3, 7, 8, 256, 90, 8, 700),
])
def test_hca_attend_matches_oracle(dtype, B, n_q, n_h, c, N, m, q_pos0):
    q, kc, vc = _attn_inputs(33, B, n_q, n_h, c, N, dtype, distinct_v=(dtype == torch.float32))
    scale = 1 / math.sqrt(c)
    o, lse = ops.hca_attend(q.to(DEV), kc.to(DEV), vc.to(DEV), m=m, q_pos0=q_pos0, scale=scale)
    ro, rl = oracle.hca_attend(q, kc, vc, m=m, q_pos0=q_pos0, scale=scale)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_out_close(to_np(o), ro, tol)
    assert max_abs(to_np(lse), rl) <= tol


@pytest.mark.parametrize("dtype,B,n_q,n_h,c,n_win,kv_pos0,n_kv,q_pos0,with_c", [
    (torch.float32, 1, 256, 4, 64, 16, 0, 256, 0, True),
    (torch.bfloat16, 2, 1, 64, 512, 128, 65536 - 128, 128, 65535, True),
    (torch.bfloat16, 1, 5, 128, 512, 128, 0, 300, 3, True),   # windows cut by the sequence start
    (torch.float32, 2, 3, 8, 128, 20, 50, 80, 110, False),    # no compressed branch
])
def test_swa_merge_matches_oracle(dtype, B, n_q, n_h, c, n_win, kv_pos0, n_kv, q_pos0, with_c):
    g = _gen(34)
    q = _randn(g, (B, n_q, n_h, c), dtype)
    kw = _randn(g, (B, n_kv, c), dtype, 1 / math.sqrt(c) * 4)
    vw = _randn(g, (B, n_kv, c), dtype)
    o_in = _randn(g, (B, n_q, n_h, c)) if with_c else None
    lse_in = _randn(g, (B, n_q, n_h)) * 3 if with_c else None
    if with_c:
        lse_in[0, 0, 0] = -math.inf  # an empty compressed set
    scale = 1 / math.sqrt(c)
    dev = lambda t: None if t is None else t.to(DEV)
    out, lse = ops.swa_merge(q.to(DEV), kw.to(DEV), vw.to(DEV), kv_pos0=kv_pos0, q_pos0=q_pos0, n_win=n_win,
                             scale=scale, o_in=dev(o_in), lse_in=dev(lse_in), out_dtype=torch.float32, want_lse=True)
    zo = np.zeros((B, n_q, n_h, c)) if o_in is None else o_in.double().numpy()
    zl = np.full((B, n_q, n_h), -np.inf) if lse_in is None else lse_in.double().numpy()
    ro, rl = oracle.swa_merge(q, kw, vw, kv_pos0, q_pos0, n_win, scale, zo, zl)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_out_close(to_np(out), ro, tol)
    assert max_abs(to_np(lse), rl) <= tol


def test_bad_index_is_skipped_and_reported():
    q, kc, vc = _attn_inputs(35, 1, 2, 8, 64, 50, torch.float32)
    idx = torch.tensor([[[1, 5, 77, -1], [2, 3, -7, 9]]], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = ops.csa_attend(q.to(DEV), kc.to(DEV), vc.to(DEV), idx.to(DEV), scale=0.2, dev_status=status)
    assert status.item() & 0x1
    clean = torch.tensor([[[1, 5, -1, -1], [2, 3, 9, -1]]], dtype=torch.int32)
    ro, _ = oracle.csa_attend(q, kc, vc, clean, 0.2)
    assert_out_close(to_np(o), ro, TOL_F32)


# ------------------------------------------------------------- end to end


def test_tiny_forward_end_to_end_matches_the_oracle_chain():
    """The float32 tiny workload (CSA + HCA + window, causal, 256 queries) run
    through HybridStep against the oracle's own chain."""
    w = workloads.WORKLOADS["tiny_f32"]
    x = workloads.make_inputs(w, "cpu")
    step = pipeline.HybridStep(w, {k: v.to(DEV) for k, v in x.items()})
    step.run()
    torch.cuda.synchronize()
    assert step.dev_status.item() == 0
    n = w.n_ctx
    # CSA layer
    ent = oracle.compress(x["ca"], x["za"], x["bias"], w.m, cb=x["cb"], zb=x["zb"], overlap=True)
    kI = oracle.compress(x["kIa"], x["zIa"], x["biasI"], w.m, cb=x["kIb"], zb=x["zIb"], overlap=True)
    assert max_abs(to_np(step.buf["entries"]), ent) <= 1e-5
    assert max_abs(to_np(step.buf["kI"]), kI) <= 1e-5
    s = oracle.index_scores(x["qI"], x["w"], kI.astype(np.float32), m=w.m, q_pos0=0)
    gidx = step.buf["idx"].cpu().numpy()
    for j in range(n):
        check_topk_row(gidx[0, j], s[0, j], oracle.visible(j, w.m), w.k)
    # the rest of the chain with the GPU's selection (identical wherever the set is unique)
    e32 = ent.astype(np.float32)
    o, l = oracle.csa_attend(x["q"], e32, e32, gidx, w.scale)
    out, _ = oracle.swa_merge(x["q"], x["kv"], x["kv"], 0, 0, w.n_win, w.scale, o, l)
    assert_out_close(to_np(step.buf["out"]), out, TOL_F32)
    # HCA layer
    eh = oracle.compress(x["ch"], x["zh"], x["bias_h"], w.m_hca).astype(np.float32)
    o, l = oracle.hca_attend(x["q"], eh, eh, m=w.m_hca, q_pos0=0, scale=w.scale)
    out, _ = oracle.swa_merge(x["q"], x["kv"], x["kv"], 0, 0, w.n_win, w.scale, o, l)
    assert_out_close(to_np(step.buf["out_h"]), out, TOL_F32)
