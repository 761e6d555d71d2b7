"""Full-size parity: the benchmark workloads run through HybridStep at their
full sizes, in the launch configuration the benchmark times, checked against
the oracle on sampled query rows (stage by stage: each oracle stage is fed the
tensors the GPU stored for the previous one).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, assert_out_close, check_topk_row, max_abs, to_np

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from sparse_attention_gated_b300 import pipeline, workloads

DEV = "cuda"


def _run(name, proj=None, **changes):
    w = workloads.WORKLOADS[name]
    if changes:
        w = workloads.scaled(w, **changes)
    x = workloads.make_inputs(w, DEV)
    cache_before = {k: x[k].clone() for k in ("kc", "kI", "kI_scale", "kc_h") if k in x}
    step = pipeline.HybridStep(w, x, proj=proj)
    step.run()
    torch.cuda.synchronize()
    assert step.dev_status.item() == 0
    return w, x, step, cache_before


def _bf16_close(got, ref):
    return max_abs(got, ref) <= 2.0 ** -7 * max(np.abs(ref).max(), 1e-3)


def _check_decode_csa(w, x, step, before, b):
    sl = slice(b, b + 1)
    cpu = lambda k: x[k][sl].cpu()
    N = w.n_csa
    t = w.n_ctx - 1
    # compress: the entry of the block ending at t lands in slot N-1, nothing else changes
    ref = oracle.compress(cpu("ca"), cpu("za"), x["bias"].cpu(), w.m, cb=cpu("cb"), zb=cpu("zb"), overlap=True,
                          first_block=N - 2)
    assert _bf16_close(to_np(x["kc"][b, N - 1]), ref[0, 0])
    assert torch.equal(x["kc"][b, : N - 1], before["kc"][b, : N - 1])
    refk = oracle.compress(cpu("kIa"), cpu("zIa"), x["biasI"].cpu(), w.m, cb=cpu("kIb"), zb=cpu("zIb"), overlap=True,
                           first_block=N - 2)[0, 0]
    dec = to_np(x["kI"][b, N - 1]) * x["kI_scale"][b, N - 1].item()
    assert np.all(np.abs(dec - refk) <= np.abs(refk) * 2.0 ** -3 + x["kI_scale"][b, N - 1].item() * 2.0 ** -9)
    # index + top-k over all N entries (the GPU's cache, including the new slot)
    s = oracle.index_scores(cpu("qI"), cpu("w"), cpu("kI"), m=w.m, q_pos0=t, qI_scale=cpu("qI_scale"),
                            kI_scale=cpu("kI_scale"))
    gidx = step.buf["idx"][sl].cpu().numpy()
    check_topk_row(gidx[0, 0], s[0, 0], N, w.k)
    # attention with the GPU's selection, then the window merge
    kc = cpu("kc")
    o, l = oracle.csa_attend(cpu("q"), kc, kc, gidx, w.scale)
    out, lu = oracle.swa_merge(cpu("q"), cpu("kv"), cpu("kv"), w.n_ctx - w.n_win, t, w.n_win, w.scale, o, l)
    assert_out_close(to_np(step.buf["out"][sl]), out)
    # the fused window merge leaves the union's lse (and no compressed-only o)
    assert max_abs(to_np(step.buf["lse"][sl]), lu) <= TOL_BF16


def _check_decode_hca(w, x, step, before, b, sfx, qkv_sfx=None):
    """qkv_sfx: suffix of the branch's queries and window rows (the cache's suffix unless
    the branch shares the CSA branch's queries, as in the parallel composition)."""
    qkv_sfx = sfx if qkv_sfx is None else qkv_sfx
    sl = slice(b, b + 1)
    cpu = lambda k: x[k][sl].cpu()
    Nh = w.n_hca
    t = w.n_ctx - 1
    kc_key = "kc" + sfx
    ref = oracle.compress(cpu("ch"), cpu("zh"), x["bias_h"].cpu(), w.m_hca, first_block=Nh - 1)
    assert _bf16_close(to_np(x[kc_key][b, Nh - 1]), ref[0, 0])
    assert torch.equal(x[kc_key][b, : Nh - 1], before[kc_key][b, : Nh - 1])
    kc = cpu(kc_key)
    q = cpu("q" + qkv_sfx)
    o, l = oracle.hca_attend(q, kc, kc, m=w.m_hca, q_pos0=t, scale=w.scale)
    kv = cpu("kv" + qkv_sfx)
    out, lu = oracle.swa_merge(q, kv, kv, w.n_ctx - w.n_win, t, w.n_win, w.scale, o, l)
    assert_out_close(to_np(step.buf["out_h"][sl]), out)
    assert max_abs(to_np(step.buf["lse_h"][sl]), lu) <= TOL_BF16


def test_flash_csa_decode_full_size():
    w, x, step, before = _run("flash_csa_decode")
    for b in (0, w.batch - 1):
        _check_decode_csa(w, x, step, before, b)


def test_flash_hca_decode_full_size():
    w, x, step, before = _run("flash_hca_decode")
    for b in (0, w.batch - 1):
        _check_decode_hca(w, x, step, before, b, "")


def test_pro_1m_hybrid_decode_full_size():
    w, x, step, before = _run("pro_1m_hybrid_decode")
    for b in (0, w.batch - 1):
        _check_decode_csa(w, x, step, before, b)
        _check_decode_hca(w, x, step, before, b, "_h")


def test_pro_1m_hybrid_decode_full_size_unit_scale_values():
    """The 1M decode with cache and window rows N(0,1) and queries N(0,2): outputs of
    order 0.1-1, so that the split join (16 splits + the window at 1M context) and
    the gathered CSA path are checked well above any rounding floor."""
    w, x, step, before = _run("pro_1m_hybrid_decode", kv_std=1.0, q_std=2.0)
    assert float(step.buf["out_h"].abs().max()) > 0.1 and float(step.buf["out"].abs().max()) > 0.1
    for b in (0, w.batch - 1):
        _check_decode_csa(w, x, step, before, b)
        _check_decode_hca(w, x, step, before, b, "_h")


def _check_in_branch(w, x, step, q0, b, layer):
    """One branch of the in-branch step for sequence b: the completed entry and the queries
    RMS-normalised and rotated at the query's position, then the attention (with the window
    merged) and the branch's sink, each stage fed the tensors the GPU stored before it."""
    sl = slice(b, b + 1)
    cpu = lambda k: x[k][sl].cpu()
    t = w.n_ctx - 1
    sfx = "" if layer == "csa" else "_h"
    if layer == "csa":
        N, kc_key = w.n_csa, "kc"
        ent = oracle.compress(cpu("ca"), cpu("za"), x["bias"].cpu(), w.m, cb=cpu("cb"), zb=cpu("zb"), overlap=True,
                              first_block=N - 2)[0, 0]
    else:
        N, kc_key = w.n_hca, "kc_h"
        ent = oracle.compress(cpu("ch"), cpu("zh"), x["bias_h"].cpu(), w.m_hca, first_block=N - 1)[0, 0]
    ent = oracle.rope_partial(oracle.rmsnorm(ent), t)
    assert _bf16_close(to_np(x[kc_key][b, N - 1]), ent)
    qn = oracle.rope_partial(oracle.rmsnorm(to_np(q0[sl])), t)
    assert _bf16_close(to_np(x["q" + sfx][sl]), qn)
    q, kc, kv = cpu("q" + sfx), cpu(kc_key), cpu("kv" + sfx)
    if layer == "csa":
        gidx = step.buf["idx"][sl].cpu().numpy()
        s = oracle.index_scores(cpu("qI"), cpu("w"), cpu("kI"), m=w.m, q_pos0=t, qI_scale=cpu("qI_scale"),
                                kI_scale=cpu("kI_scale"))
        check_topk_row(gidx[0, 0], s[0, 0], N, w.k)
        o, l = oracle.csa_attend(q, kc, kc, gidx, w.scale)
    else:
        o, l = oracle.hca_attend(q, kc, kc, m=w.m_hca, q_pos0=t, scale=w.scale)
    out, lu = oracle.swa_merge(q, kv, kv, w.n_ctx - w.n_win, t, w.n_win, w.scale, o, l)
    out, lu = oracle.sink_merge(out, lu, x["sink" + sfx].cpu())
    assert_out_close(to_np(step.buf["out" + sfx][sl]), out)
    assert max_abs(to_np(step.buf["lse" + sfx][sl]), lu) <= TOL_BF16


def test_pro_1m_hybrid_decode_in_branch_full_size():
    """The 1M hybrid decode with the in-branch operations as the benchmark times them:
    RMSNorm + partial RoPE of both layers' queries and completed entries, and each
    layer's per-head attention sink on its merged result."""
    w = workloads.WORKLOADS["pro_1m_hybrid_decode_in_branch"]
    x = workloads.make_inputs(w, DEV)
    q0, q0_h = x["q"].clone(), x["q_h"].clone()
    step = pipeline.HybridStep(w, x)
    step.run()
    torch.cuda.synchronize()
    assert step.dev_status.item() == 0
    for b in (0, w.batch - 1):
        _check_in_branch(w, x, step, q0, b, "csa")
        _check_in_branch(w, x, step, q0_h, b, "hca")


def _proj_weights(seed, g, d_g, k):
    gen = torch.Generator()
    gen.manual_seed(seed)
    return (torch.randn((g, d_g, k), generator=gen) / math.sqrt(k)).to(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("kv_std,q_std", [(None, 1.0), (1.0, 2.0)])
def test_pro_1m_parallel_decode_full_size_with_grouped_projection(kv_std, q_std):
    """CSA and HCA side by side on the same queries and window, at 1M context: each branch
    against the oracle chain, then the grouped projection of the 2 n_h concatenated heads
    (16 groups of 16 heads; the first 8 groups read the CSA heads) fed the GPU's outputs."""
    w0 = workloads.WORKLOADS["pro_1m_parallel_decode"]
    g, d_g = 16, 256
    W = _proj_weights(83, g, d_g, 2 * w0.n_h * w0.c // g)
    w, x, step, before = _run("pro_1m_parallel_decode", proj=dict(w=W), kv_std=kv_std, q_std=q_std)
    for b in (0, w.batch - 1):
        _check_decode_csa(w, x, step, before, b)
        _check_decode_hca(w, x, step, before, b, "_h", qkv_sfx="")
    cat = torch.cat([step.buf["out"], step.buf["out_h"]], dim=-2)
    ref = oracle.grouped_out_proj(to_np(cat), W.double().cpu().numpy())
    assert_out_close(to_np(step.buf["proj"]), ref, tol=1e-3, rel=1e-3, what="projection")


@pytest.mark.parametrize("kv_std,q_std", [(None, 1.0), (1.0, 2.0)])
def test_flash_swa_decode_full_size(kv_std, q_std):
    """A pure sliding-window layer (Flash shapes): softmax attention over the window alone."""
    w, x, step, _ = _run("flash_swa_decode", kv_std=kv_std, q_std=q_std)
    t = w.n_ctx - 1
    for b in (0, w.batch - 1):
        sl = slice(b, b + 1)
        q, kv = x["q"][sl].cpu(), x["kv"][sl].cpu()
        shape = q.shape[:3]
        out, _ = oracle.swa_merge(q, kv, kv, w.n_ctx - w.n_win, t, w.n_win, w.scale, np.zeros(q.shape),
                                  np.full(shape, -np.inf))
        assert_out_close(to_np(step.buf["out"][sl]), out)


def test_flash_decodes_full_size_unit_scale_values():
    for name, check in (("flash_csa_decode", _check_decode_csa), ("flash_hca_decode", _check_decode_hca)):
        w, x, step, before = _run(name, kv_std=1.0, q_std=2.0)
        for b in (0, w.batch - 1):
            if check is _check_decode_hca:
                check(w, x, step, before, b, "")
            else:
                check(w, x, step, before, b)


def test_csa_prefill_unit_scale_values_sampled_rows():
    """A prefill chunk of 8,192 tokens (Pro shapes) with unit-scale rows: query tiles,
    the causal edge and the two-launch window merge with O(1) outputs."""
    _check_prefill(*_run("pro_csa_prefill", n_ctx=8192, kv_std=1.0, q_std=2.0)[:3],
                   rows=(0, 3, 4, 127, 128, 1000, 4095, 4096, 8191))


def test_pro_csa_prefill_full_size_sampled_rows():
    _check_prefill(*_run("pro_csa_prefill")[:3], rows=(0, 2, 3, 4, 127, 128, 4095, 4096, 16383, 32767))


def _check_prefill(w, x, step, rows):
    cpu = {k: v.cpu() for k, v in x.items()}
    ent = oracle.compress(cpu["ca"], cpu["za"], cpu["bias"], w.m, cb=cpu["cb"], zb=cpu["zb"], overlap=True)
    assert _bf16_close(to_np(step.buf["entries"]), ent)
    refk = oracle.compress(cpu["kIa"], cpu["zIa"], cpu["biasI"], w.m, cb=cpu["kIb"], zb=cpu["zIb"], overlap=True)
    sc = step.buf["kI_scale"].cpu().numpy()[..., None]
    dec = to_np(step.buf["kI"]) * sc
    assert np.all(np.abs(dec - refk) <= np.abs(refk) * 2.0 ** -3 + sc * 2.0 ** -9)
    kI, kIs = step.buf["kI"].cpu(), step.buf["kI_scale"].cpu()
    e = step.buf["entries"].cpu()
    gidx = step.buf["idx"].cpu().numpy()
    for j in rows:
        js = slice(j, j + 1)
        s = oracle.index_scores(cpu["qI"][:, js], cpu["w"][:, js], kI, m=w.m, q_pos0=j,
                                qI_scale=cpu["qI_scale"][:, js], kI_scale=kIs)
        check_topk_row(gidx[0, j], s[0, 0], oracle.visible(j, w.m), w.k)
        o, l = oracle.csa_attend(cpu["q"][:, js], e, e, gidx[:, js], w.scale)
        out, lu = oracle.swa_merge(cpu["q"][:, js], cpu["kv"], cpu["kv"], 0, j, w.n_win, w.scale, o, l)
        assert_out_close(to_np(step.buf["out"][:, js]), out)
        assert max_abs(to_np(step.buf["lse"][:, js]), lu) <= TOL_BF16
