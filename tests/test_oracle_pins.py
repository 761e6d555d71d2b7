"""Pins of the float64 oracle to things other than itself.

Each test checks the oracle against a value printed on the pages (with its
citation), a closed form, a special case that reduces to a library routine
(numpy / torch), or brute force on tiny inputs.  These run on CPU only.

Pages cited:
  [HA]  "DeepSeek-V4 hybrid attention: CSA, HCA, mHC, MoE" (trishampatil.com)
  [DV4] "DeepSeek-V4: Anatomy of an Open-Source Frontier Model" (modernaiengineering.com)
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ formats


def test_bf16_decode_is_upper_half_of_binary32():
    bits = _rng(1).integers(0, 1 << 16, 4000, dtype=np.uint32).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_decode(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == 448.0  # largest finite


def test_e4m3_encode_matches_torch_round_to_nearest_even():
    rng = _rng(2)
    x = np.concatenate([rng.normal(0, 1, 3000), rng.uniform(-448, 448, 3000), rng.normal(0, 1e-2, 1000)])
    # exact midpoints between neighbouring positive codes exercise the tie rule
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([x, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    assert oracle.e4m3_encode(np.array([1e6, -1e6, 449.0, 470.0], dtype=np.float32)).tolist() == [0x7E, 0xFE, 0x7E,
                                                                                                   0x7E]


def test_round_bf16_matches_torch_from_float32():
    x = _rng(3).normal(0, 10, 5000).astype(np.float32)
    x[:10] = [0.0, 1e-40, -1e-39, 3.0e38, 1.0, -2.5, 1.00390625, 1.01171875, 65504.0, 1e-30]
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------- counts


def test_entry_counts_printed_for_one_million_tokens():
    """[DV4] csa_hca_budget.py output: stored / attended entries at n = 1,000,000."""
    g = _golden("csa_hca_budget.json")
    n = g["n"]
    m, mh, k, win = g["m_csa"], g["m_hca"], g["top_k"], g["window"]
    t = n - 1
    n_csa = oracle.compress_out_count(n, m, overlap=True)
    n_hca = oracle.compress_out_count(n, mh, overlap=False)
    # top-k count: run the selector on the n/m visible entries
    scores = _rng(4).random((1, n_csa))
    sel = oracle.topk(scores, [oracle.visible(t, m)], k)
    attended_csa = int((sel >= 0).sum()) + oracle.window_count(t, win)
    stored_csa = n_csa + oracle.window_count(t, win)
    stored_hca = oracle.visible(t, mh) + oracle.window_count(t, win)
    assert stored_csa == g["table"]["CSA"]["stored"]
    assert attended_csa == g["table"]["CSA"]["attended"]
    assert stored_hca == g["table"]["HCA"]["stored"] == g["table"]["HCA"]["attended"]


def test_entry_counts_worked_example_three_context_sizes():
    """[DV4] worked example: a CSA query reads 628 / 1,152 / 1,152 entries at
    n = 2,000 / 32,000 / 1,000,000 (Pro settings: m = 4, top-k 1,024, window 128)."""
    g = _golden("worked_example_counts.json")
    for row in g["rows"]:
        n = row["n"]
        t = n - 1
        vis = oracle.visible(t, 4)
        scores = _rng(5).random((1, vis))
        sel = oracle.topk(scores, [vis], 1024)
        assert int((sel >= 0).sum()) + oracle.window_count(t, 128) == row["attended"]


# ----------------------------------------------------------------- compress


def _csa_inputs(seed, B=2, n=40, c=6, m=4):
    r = _rng(seed)
    f = lambda *s: r.normal(0, 1, s).astype(np.float32)
    return f(B, n, c), f(B, n, c), f(B, n, c), f(B, n, c), f(2 * m, c)


def test_pooling_weights_sum_to_one():
    ca, cb, za, zb, bias = _csa_inputs(6)
    for j, ch in [(0, 0), (3, 2), (9, 5)]:
        w = oracle.compress_weights(za, bias, 4, b=1, j=j, ch=ch, zb=zb, overlap=True)
        assert abs(w.sum() - 1.0) < 1e-12 and (w >= 0).all()
    w = oracle.compress_weights(za, bias[:4], 4, b=0, j=2, ch=1, overlap=False)
    assert abs(w.sum() - 1.0) < 1e-12


def test_constant_values_pool_to_the_constant():
    ca, cb, za, zb, bias = _csa_inputs(7)
    const = np.full_like(ca, 0.75)
    out = oracle.compress(const, za, bias, 4, cb=const, zb=zb, overlap=True)
    assert np.allclose(out, 0.75, atol=1e-14, rtol=0)


def test_uniform_gates_give_the_block_mean():
    """With Z constant and no bias the gate is uniform: the entry is np.mean of its block."""
    ca, _, _, _, _ = _csa_inputs(8, n=64, c=5)
    z = np.zeros_like(ca)
    for m in (1, 4, 16):
        out = oracle.compress(ca, z, np.zeros((m, 5), np.float32), m)
        ref = ca.astype(np.float64).reshape(2, 64 // m, m, 5).mean(axis=2)
        assert np.allclose(out, ref, atol=1e-13, rtol=0)


def test_one_hot_gate_pins_the_overlap_geometry():
    """[HA] V.1: entry i draws on stream a of block i and stream b of block i-1.
    A dominant logit on one raw row makes the entry equal that row's value."""
    B, n, c, m = 1, 24, 3, 4
    r = _rng(9)
    ca = r.normal(0, 1, (B, n, c)).astype(np.float32)
    cb = r.normal(0, 1, (B, n, c)).astype(np.float32)
    for row in (0, 5, 11, 23):
        for stream in ("a", "b"):
            za = np.zeros((B, n, c), np.float32)
            zb = np.zeros((B, n, c), np.float32)
            (za if stream == "a" else zb)[0, row, 1] = 80.0
            out = oracle.compress(ca, za, np.zeros((2 * m, c), np.float32), m, cb=cb, zb=zb, overlap=True)
            entry = row // m if stream == "a" else row // m + 1
            if entry >= n // m:
                continue
            src = ca if stream == "a" else cb
            assert abs(out[0, entry, 1] - src[0, row, 1]) < 1e-12


def test_one_hot_bias_pins_the_position_layout():
    """Bias row p < m weights stream b of the previous block; row m + p weights stream a."""
    B, n, c, m = 1, 20, 2, 4
    r = _rng(10)
    ca = r.normal(0, 1, (B, n, c)).astype(np.float32)
    cb = r.normal(0, 1, (B, n, c)).astype(np.float32)
    z = np.zeros((B, n, c), np.float32)
    for p in range(2 * m):
        bias = np.zeros((2 * m, c), np.float32)
        bias[p, :] = 80.0
        out = oracle.compress(ca, z, bias, m, cb=cb, zb=z, overlap=True)
        for i in range(1, n // m):
            want = cb[0, (i - 1) * m + p] if p < m else ca[0, i * m + (p - m)]
            assert np.allclose(out[0, i], want, atol=1e-12, rtol=0)


def test_first_entry_has_no_previous_block():
    """Entry 0 pools stream a only, whatever stream b says (reading R3)."""
    ca, cb, za, zb, bias = _csa_inputs(11, n=16)
    zb_big = zb + 100.0
    out = oracle.compress(ca, za, bias, 4, cb=cb, zb=zb_big, overlap=True)
    alone = oracle.compress(ca, za, bias[4:], 4)  # HCA form over stream a with the stream-a bias rows
    assert np.allclose(out[:, 0], alone[:, 0], atol=1e-12)
    # later entries are (almost) pure stream b of the previous block
    prev_b = oracle.compress(cb, zb_big, bias[:4], 4)
    assert np.allclose(out[:, 1:], prev_b[:, :-1], atol=1e-12)


def test_append_form_matches_full_compress():
    """Compressing two blocks with first_block = i-1 yields entry i of the full run."""
    ca, cb, za, zb, bias = _csa_inputs(12, n=32)
    full = oracle.compress(ca, za, bias, 4, cb=cb, zb=zb, overlap=True)
    for i in (1, 3, 7):
        sl = slice((i - 1) * 4, (i + 1) * 4)
        one = oracle.compress(ca[:, sl], za[:, sl], bias, 4, cb=cb[:, sl], zb=zb[:, sl], overlap=True, first_block=i - 1)
        # block 0 has no predecessor, so it is an entry of its own; any other first block only feeds the next
        assert one.shape[1] == (2 if i == 1 else 1)
        assert np.array_equal(one[:, -1], full[:, i])


def test_budget_toy_indexer_picks_blocks_0_and_1():
    """[DV4] csa_hca_budget.py (np.random.seed(0)): 16 tokens -> 4 entries with
    softmax position weights; the indexer picks compressed blocks [0, 1]."""
    g = _golden("csa_hca_budget.json")
    np.random.seed(0)
    m, d = 4, 6
    keys = np.random.randn(16, d)
    w_logits = np.random.randn(m)
    q = np.random.randn(d)
    # position weights as the gate: Z = 0, bias[p][:] = w_logits[p]
    bias = np.repeat(w_logits[:, None], d, axis=1).astype(np.float32)
    k32 = keys[None].astype(np.float32)
    comp = oracle.compress(k32, np.zeros_like(k32), bias, m)
    assert comp.shape[1] == g["compressed_entries"]
    # one indexer head with weight 1: I = ReLU(q . k)
    s = oracle.index_scores(q[None, None, None].astype(np.float32), np.ones((1, 1, 1), np.float32),
                            comp.astype(np.float32), m=1, q_pos0=10 ** 6)
    idx = oracle.topk(s, [4], 2)[0, 0]
    ranked = sorted(idx.tolist(), key=lambda e: -s[0, 0, e])
    assert ranked == g["indexer_picks"]


def test_pooling_recall_toy_printed_output():
    """[DV4] practice_pooling_recall.py (default_rng(0)): mean pooling x1/x4/x16."""
    g = _golden("pooling_recall.json")
    rng = np.random.default_rng(0)
    n, d = 64, 8
    keys = rng.normal(0, 1, (n, d))
    needle = 37
    query = keys[needle] + rng.normal(0, 0.3, d)
    k32 = keys[None].astype(np.float32)
    q32 = query[None, None, None].astype(np.float32)
    for row in g["rows"]:
        m = row["m"]
        ent = oracle.compress(k32, np.zeros_like(k32), np.zeros((m, d), np.float32), m)
        s = oracle.index_scores(q32, np.ones((1, 1, 1), np.float32), ent.astype(np.float32), m=1, q_pos0=10 ** 6)[0, 0]
        assert ent.shape[1] == row["entries"]
        best = int(oracle.topk(s[None], [len(s)], 1)[0, 0])
        assert best == row["best_entry"]
        assert (best == needle // m) == row["holds_needle"]
        top2 = sorted(s)[-2:]
        assert round(top2[1] - top2[0], 2) == row["lead"]
    ent = oracle.compress(k32, np.zeros_like(k32), np.zeros((4, d), np.float32), 4)
    s = oracle.index_scores(q32, np.ones((1, 1, 1), np.float32), ent.astype(np.float32), m=1, q_pos0=10 ** 6)[0, 0]
    sel = oracle.topk(s[None], [16], g["top_k"])[0]
    assert sorted(sel.tolist(), key=lambda e: -s[e]) == g["topk_x4"]
    assert g["top_k"] + oracle.window_count(n - 1, g["window"]) == g["entries_attended"]


# ----------------------------------------------------------------- quantise


def test_quantiser_matches_library_cast_of_scaled_rows():
    x = _rng(13).normal(0, 1, (50, 128)).astype(np.float32)
    x[3] = 0.0
    codes, scales = oracle.quantise_fp8_rows(x)
    amax = np.abs(x).max(axis=1)
    exp_scale = np.where(amax > 0, (amax / np.float32(448)).astype(np.float32), np.float32(1))
    assert np.array_equal(scales, exp_scale)
    y = (torch.from_numpy(x) / torch.from_numpy(exp_scale)[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(codes, y.numpy())
    # the row maximum lands exactly on +-448
    i = np.abs(x[0]).argmax()
    assert abs(oracle.e4m3_decode(codes[0, i : i + 1])[0]) == 448.0


# -------------------------------------------------------------------- index


def test_single_head_unit_weight_index_is_relu_of_dot():
    r = _rng(14)
    q = r.normal(0, 1, (1, 3, 1, 8)).astype(np.float32)
    k = r.normal(0, 1, (1, 12, 8)).astype(np.float32)
    s = oracle.index_scores(q, np.ones((1, 3, 1), np.float32), k, m=1, q_pos0=100)
    ref = np.maximum(np.einsum("jd,sd->js", q[0, :, 0].astype(np.float64), k[0].astype(np.float64)), 0)
    assert np.allclose(s[0], ref, atol=1e-12, rtol=0)


def test_index_is_weighted_sum_over_heads():
    """Multi-head score = sum over heads of single-head scores times w[t,h]."""
    r = _rng(15)
    q = r.normal(0, 1, (2, 3, 4, 8)).astype(np.float32)
    k = r.normal(0, 1, (2, 10, 8)).astype(np.float32)
    w = r.uniform(0, 1, (2, 3, 4)).astype(np.float32)
    full = oracle.index_scores(q, w, k, m=1, q_pos0=50)
    acc = np.zeros_like(full)
    for h in range(4):
        acc += w[:, :, h, None].astype(np.float64) * oracle.index_scores(
            np.ascontiguousarray(q[:, :, h : h + 1]), np.ones((2, 3, 1), np.float32), k, m=1, q_pos0=50)
    assert np.allclose(full, acc, atol=1e-12, rtol=0)


def test_fp8_index_equals_float_index_on_decoded_values():
    r = _rng(16)
    q8 = torch.from_numpy(r.normal(0, 1, (1, 2, 4, 16)).astype(np.float32)).to(torch.float8_e4m3fn)
    k8 = torch.from_numpy(r.normal(0, 1, (1, 9, 16)).astype(np.float32)).to(torch.float8_e4m3fn)
    # scales with few significant bits keep code x scale exact in float32
    qs = r.choice([0.5, 0.75, 1.0, 1.25, 1.5, 2.0], (1, 2, 4)).astype(np.float32)
    ks = r.choice([0.5, 0.75, 1.0, 1.25, 1.5, 2.0], (1, 9)).astype(np.float32)
    w = r.uniform(0, 1, (1, 2, 4)).astype(np.float32)
    s8 = oracle.index_scores(q8, w, k8, m=1, q_pos0=40, qI_scale=qs, kI_scale=ks)
    qf = (q8.to(torch.float64).numpy() * qs[..., None]).astype(np.float32)
    kf = (k8.to(torch.float64).numpy() * ks[..., None]).astype(np.float32)
    sf = oracle.index_scores(qf, w, kf, m=1, q_pos0=40)
    assert np.allclose(s8, sf, atol=1e-12, rtol=1e-12)


def test_index_sees_only_completed_blocks():
    """Reading R5: entry s is visible at position t iff its last token m(s+1)-1 <= t."""
    r = _rng(17)
    m, N = 4, 8
    q = r.normal(0, 1, (1, 32, 1, 4)).astype(np.float32)
    k = r.normal(0, 1, (1, N, 4)).astype(np.float32)
    s = oracle.index_scores(q, np.ones((1, 32, 1), np.float32), k, m=m, q_pos0=0)
    for t in range(32):
        for e in range(N):
            last_token = m * (e + 1) - 1
            assert np.isfinite(s[0, t, e]) == (last_token <= t)


# -------------------------------------------------------------------- top-k


def test_topk_is_the_max_sum_subset_brute_force():
    r = _rng(18)
    for trial in range(40):
        V = int(r.integers(1, 10))
        k = int(r.integers(1, 5))
        s = r.normal(0, 1, V)
        got = oracle.topk(s[None], [V], k)[0]
        take = min(k, V)
        best = max(itertools.combinations(range(V), take), key=lambda c: sum(s[i] for i in c))
        assert got[:take].tolist() == sorted(best)
        assert (got[take:] == -1).all()


def test_topk_agrees_with_numpy_argsort_and_respects_visibility():
    r = _rng(19)
    s = r.normal(0, 1, (6, 300))
    vis = np.array([0, 1, 17, 128, 299, 300])
    got = oracle.topk(s, vis, 64)
    for row in range(6):
        v = vis[row]
        ref = np.sort(np.argsort(-s[row, :v], kind="stable")[: min(64, v)])
        n_valid = min(64, v)
        assert got[row, :n_valid].tolist() == ref.tolist()
        assert (got[row, n_valid:] == -1).all()


def test_topk_ties_go_to_the_lower_index():
    s = np.zeros((1, 10))
    assert oracle.topk(s, [10], 3)[0].tolist() == [0, 1, 2]
    s = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]])
    assert oracle.topk(s, [5], 2)[0].tolist() == [1, 2]


# ---------------------------------------------------------------- attention


def _sdpa(q, k, v, mask, scale):
    """Reference: torch scaled_dot_product_attention in float64 (a library routine)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=torch.from_numpy(mask),
        scale=scale).numpy()


def test_m1_uniform_hca_reduces_to_causal_mqa():
    """With m' = 1 and uniform gates each entry is a raw row, so the compressed
    branch is plain causal multi-query attention over the raw rows."""
    r = _rng(20)
    B, n, H, c = 1, 24, 3, 8
    kv = r.normal(0, 1, (B, n, c)).astype(np.float32)
    q = r.normal(0, 1, (B, n, H, c)).astype(np.float32)
    ent = oracle.compress(kv, np.zeros_like(kv), np.zeros((1, c), np.float32), 1).astype(np.float32)
    scale = 1 / math.sqrt(c)
    o, lse = oracle.hca_attend(q, ent, ent, m=1, q_pos0=0, scale=scale)
    qh = q.astype(np.float64).transpose(0, 2, 1, 3)  # B H n c
    kk = np.repeat(kv.astype(np.float64)[:, None], H, axis=1)
    mask = np.tril(np.ones((n, n), dtype=bool))
    ref = _sdpa(qh, kk, kk, mask, scale).transpose(0, 2, 1, 3)
    assert np.allclose(o, ref, atol=1e-12)
    logits = np.einsum("bthc,bsc->bths", q.astype(np.float64), kv.astype(np.float64)) * scale
    logits = np.where(mask[None, :, None, :], logits, -np.inf)
    ref_lse = torch.logsumexp(torch.from_numpy(logits), dim=-1).numpy()
    assert np.allclose(lse, ref_lse, atol=1e-12)


def test_m1_csa_with_full_topk_reduces_to_causal_mqa():
    """CSA form with m = 1, stream b switched off and k >= #entries selects every
    visible entry, so CSA attention is plain causal attention over the raw rows."""
    r = _rng(21)
    B, n, H, c, nih, cI = 1, 20, 2, 8, 3, 4
    kv = r.normal(0, 1, (B, n, c)).astype(np.float32)
    q = r.normal(0, 1, (B, n, H, c)).astype(np.float32)
    za = np.zeros_like(kv)
    zb = np.full_like(kv, -1e30)  # stream-b logits -> -inf
    ent = oracle.compress(kv, za, np.zeros((2, c), np.float32), 1, cb=kv, zb=zb, overlap=True).astype(np.float32)
    assert np.array_equal(ent, kv)
    kI = r.normal(0, 1, (B, n, cI)).astype(np.float32)
    qI = r.normal(0, 1, (B, n, nih, cI)).astype(np.float32)
    w = r.uniform(0, 1, (B, n, nih)).astype(np.float32)
    s = oracle.index_scores(qI, w, kI, m=1, q_pos0=0)
    idx = oracle.topk(s, [oracle.visible(t, 1) for t in range(n)], n)
    scale = 1 / math.sqrt(c)
    o, _ = oracle.csa_attend(q, ent, ent, idx, scale)
    qh = q.astype(np.float64).transpose(0, 2, 1, 3)
    kk = np.repeat(kv.astype(np.float64)[:, None], H, axis=1)
    ref = _sdpa(qh, kk, kk, np.tril(np.ones((n, n), dtype=bool)), scale).transpose(0, 2, 1, 3)
    assert np.allclose(o, ref, atol=1e-12)


def test_hca_is_dense_attention_over_pooled_entries():
    r = _rng(22)
    B, n, H, c, m = 2, 64, 2, 6, 8
    kv = r.normal(0, 1, (B, n, c)).astype(np.float32)
    z = r.normal(0, 1, (B, n, c)).astype(np.float32)
    bias = r.normal(0, 1, (m, c)).astype(np.float32)
    ent = oracle.compress(kv, z, bias, m).astype(np.float32)
    N = ent.shape[1]
    q = r.normal(0, 1, (B, 4, H, c)).astype(np.float32)
    q_pos0 = n - 4
    o, _ = oracle.hca_attend(q, ent, ent, m=m, q_pos0=q_pos0, scale=0.3)
    # at these positions every entry is complete: plain dense attention over all of them
    qh = q.astype(np.float64).transpose(0, 2, 1, 3)
    ee = np.repeat(ent.astype(np.float64)[:, None], H, axis=1)
    vis = np.array([[oracle.visible(q_pos0 + j, m) > s for s in range(N)] for j in range(4)])
    ref = _sdpa(qh, ee, ee, vis, 0.3).transpose(0, 2, 1, 3)
    assert np.allclose(o, ref, atol=1e-12)


def test_single_entry_set_returns_that_value():
    r = _rng(23)
    q = r.normal(0, 1, (1, 1, 2, 5)).astype(np.float32)
    k = r.normal(0, 1, (1, 7, 5)).astype(np.float32)
    v = r.normal(0, 1, (1, 7, 5)).astype(np.float32)
    idx = np.array([[[4, -1, -1]]], np.int32)
    o, lse = oracle.csa_attend(q, k, v, idx, 0.5)
    assert np.allclose(o[0, 0], np.repeat(v[0, 4:5].astype(np.float64), 2, axis=0), atol=1e-15)
    assert np.allclose(lse[0, 0], 0.5 * q[0, 0].astype(np.float64) @ k[0, 4].astype(np.float64), atol=1e-12)
    o, lse = oracle.csa_attend(q, k, v, np.full((1, 1, 3), -1, np.int32), 0.5)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_attention_weights_sum_to_one():
    """Values all equal to one vector => the output is that vector (rows of p sum to 1)."""
    r = _rng(24)
    q = r.normal(0, 3, (1, 2, 3, 4)).astype(np.float32)
    k = r.normal(0, 3, (1, 50, 4)).astype(np.float32)
    vec = r.normal(0, 1, 4).astype(np.float32)
    v = np.broadcast_to(vec, (1, 50, 4)).copy()
    idx = np.sort(r.choice(50, (1, 2, 20), replace=True), axis=-1).astype(np.int32)
    o, _ = oracle.csa_attend(q, k, v, idx, 1.0)
    assert np.allclose(o, vec.astype(np.float64), atol=1e-13)


def test_merge_equals_one_softmax_over_the_union():
    """[DV4] step 5: attend the selected entries and the window as one set."""
    r = _rng(25)
    B, H, c, N, n_kv, n_win = 1, 2, 6, 30, 40, 8
    q = r.normal(0, 1, (B, 3, H, c)).astype(np.float32)
    kc = r.normal(0, 1, (B, N, c)).astype(np.float32)
    vc = r.normal(0, 1, (B, N, c)).astype(np.float32)
    kw = r.normal(0, 1, (B, n_kv, c)).astype(np.float32)
    vw = r.normal(0, 1, (B, n_kv, c)).astype(np.float32)
    idx = np.sort(r.choice(N, (B, 3, 7), replace=False), axis=-1).astype(np.int32)
    kv_pos0, q_pos0, scale = 100, 130, 0.4
    o_c, lse_c = oracle.csa_attend(q, kc, vc, idx, scale)
    out, lse = oracle.swa_merge(q, kw, vw, kv_pos0, q_pos0, n_win, scale, o_c, lse_c)
    for j in range(3):
        t = q_pos0 + j
        rows = np.arange(t - n_win + 1, t + 1) - kv_pos0
        K = np.concatenate([kc[0, idx[0, j]], kw[0, rows]]).astype(np.float64)
        V = np.concatenate([vc[0, idx[0, j]], vw[0, rows]]).astype(np.float64)
        qh = q[0, j].astype(np.float64)[None, :, None, :]  # 1 H 1 c
        ref = _sdpa(qh, np.repeat(K[None, None], H, 1), np.repeat(V[None, None], H, 1),
                    np.ones((1, len(K)), dtype=bool), scale)[0, :, 0]
        assert np.allclose(out[0, j], ref, atol=1e-12)
        ref_lse = torch.logsumexp(torch.from_numpy(qh[0, :, 0] @ K.T * scale), dim=-1).numpy()
        assert np.allclose(lse[0, j], ref_lse, atol=1e-12)


def test_merge_with_empty_compressed_side_is_the_window_alone():
    r = _rng(26)
    q = r.normal(0, 1, (1, 2, 2, 4)).astype(np.float32)
    kw = r.normal(0, 1, (1, 10, 4)).astype(np.float32)
    o_c = np.zeros((1, 2, 2, 4))
    lse_c = np.full((1, 2, 2), -np.inf)
    out, lse = oracle.swa_merge(q, kw, kw, 0, 3, 16, 0.5, o_c, lse_c)
    for j in range(2):
        t = 3 + j
        K = kw[0, : t + 1].astype(np.float64)
        qh = q[0, j].astype(np.float64)
        p = np.exp(qh @ K.T * 0.5)
        p /= p.sum(axis=1, keepdims=True)
        assert np.allclose(out[0, j], p @ K, atol=1e-12)


def test_window_covers_exactly_the_last_n_win_rows():
    """A row just outside the window has no influence; the oldest row inside does."""
    r = _rng(27)
    q = r.normal(0, 1, (1, 1, 1, 4)).astype(np.float32)
    kw = r.normal(0, 1, (1, 40, 4)).astype(np.float32)
    o0 = np.zeros((1, 1, 1, 4))
    l0 = np.full((1, 1, 1), -np.inf)
    t, n_win = 30, 8
    base, _ = oracle.swa_merge(q, kw, kw, 0, t, n_win, 1.0, o0, l0)
    out_far = kw.copy()
    out_far[0, t - n_win] = np.nan
    out_far[0, t + 1 :] = np.nan
    far, _ = oracle.swa_merge(q, out_far, out_far, 0, t, n_win, 1.0, o0, l0)
    assert np.array_equal(far, base)
    near = kw.copy()
    near[0, t - n_win + 1] += 1.0
    moved, _ = oracle.swa_merge(q, near, near, 0, t, n_win, 1.0, o0, l0)
    assert not np.allclose(moved, base)


def test_pipeline_never_reads_the_future():
    """Poisoning every raw row after a query's position leaves its output unchanged."""
    r = _rng(28)
    B, n, c, H, m, mh, nih, cI, k, n_win = 1, 48, 6, 2, 4, 8, 2, 4, 3, 5
    f = lambda *s: r.normal(0, 1, s).astype(np.float32)
    ca, cb, za, zb, kv = f(B, n, c), f(B, n, c), f(B, n, c), f(B, n, c), f(B, n, c)
    kIa, kIb, zIa, zIb = f(B, n, cI), f(B, n, cI), f(B, n, cI), f(B, n, cI)
    bias, biasI, biash = f(2 * m, c), f(2 * m, cI), f(mh, c)
    q, qI, w = f(B, n, H, c), f(B, n, nih, cI), r.uniform(0, 1, (B, n, nih)).astype(np.float32)

    def forward(ca, cb, za, zb, kIa, kIb, zIa, zIb, kv):
        ent = oracle.compress(ca, za, bias, m, cb=cb, zb=zb, overlap=True).astype(np.float32)
        kI = oracle.compress(kIa, zIa, biasI, m, cb=kIb, zb=zIb, overlap=True).astype(np.float32)
        s = oracle.index_scores(qI, w, kI, m=m, q_pos0=0)
        idx = oracle.topk(s, [oracle.visible(t, m) for t in range(n)], k)
        o, l = oracle.csa_attend(q, ent, ent, idx, 0.4)
        csa, _ = oracle.swa_merge(q, kv, kv, 0, 0, n_win, 0.4, o, l)
        hent = oracle.compress(ca, za, biash, mh).astype(np.float32)
        o, l = oracle.hca_attend(q, hent, hent, m=mh, q_pos0=0, scale=0.4)
        hca, _ = oracle.swa_merge(q, kv, kv, 0, 0, n_win, 0.4, o, l)
        return csa, hca

    base = forward(ca, cb, za, zb, kIa, kIb, zIa, zIb, kv)
    for t in (5, 17, 31):
        poisoned = [a.copy() for a in (ca, cb, za, zb, kIa, kIb, zIa, zIb, kv)]
        for a in poisoned:
            a[:, t + 1 :] = np.nan
        got = forward(*poisoned)
        for g, b in zip(got, base):
            assert np.array_equal(g[:, : t + 1], b[:, : t + 1])


# --------------------------------------------- in-branch operations ([HA] IV)


def test_rmsnorm_rows_have_unit_rms_and_ignore_scale():
    x = _rng(61).normal(size=(7, 64)) * _rng(62).uniform(0.1, 10, size=(7, 1))
    y = oracle.rmsnorm(x, eps=0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-12)
    assert np.allclose(oracle.rmsnorm(3.5 * x, eps=0.0), y, atol=1e-12)
    assert np.allclose(oracle.rmsnorm(-x, eps=0.0), -y, atol=1e-12)


def test_rmsnorm_worked_values_and_gain():
    # [3, 4]: mean square 12.5, so the row divides by sqrt(12.5) = 3.5355...
    y = oracle.rmsnorm(np.array([[3.0, 4.0]]), eps=0.0)
    assert np.allclose(y, [[0.848528137423857, 1.131370849898476]], atol=1e-12)
    # a constant row v gives sign(v) in every channel; the gain scales channel by channel
    g = np.array([2.0, -1.0, 0.5, 4.0])
    assert np.allclose(oracle.rmsnorm(np.full((1, 4), -0.3), g, eps=0.0), -g, atol=1e-12)
    # eps enters under the root: a zero row stays zero, and x^2 mean 1 with eps 3 halves the row
    assert np.all(oracle.rmsnorm(np.zeros((1, 8)), eps=1e-6) == 0.0)
    assert np.allclose(oracle.rmsnorm(np.ones((1, 8)), eps=3.0), 0.5, atol=1e-12)


def test_partial_rope_leaves_the_leading_dims_and_pair_norms():
    x = _rng(63).normal(size=(5, 96))
    pos = np.array([0.0, 1.0, 17.0, 1000.0, 123456.0])
    y = oracle.rope_partial(x, pos, rope_dims=64)
    assert np.array_equal(y[:, :32], x[:, :32])
    assert np.allclose(y[0], x[0], atol=0)  # position 0: no rotation
    pn = lambda a: np.hypot(a[:, 32::2], a[:, 33::2])
    assert np.allclose(pn(y), pn(x), atol=1e-12)


def test_partial_rope_composes_and_depends_on_relative_position_only():
    r = _rng(64)
    q, k = r.normal(size=(1, 128)), r.normal(size=(1, 128))
    a, b = 321.0, 77.0
    rq = lambda v, p: oracle.rope_partial(v, [p], rope_dims=64)
    assert np.allclose(rq(rq(q, a), b), rq(q, a + b), atol=1e-9)
    assert np.isclose((rq(q, a) @ rq(k, b).T).item(), (rq(q, a - b) @ k.T).item(), atol=1e-9)


def test_partial_rope_frequencies_worked_values():
    # rope_dims = 4, theta = 10000: pair 0 turns by the position itself, pair 1 by
    # position * 10000^(-2/4) = position / 100; so at position 100 both turn by 1 radian
    x = np.array([[9.0, 1.0, 0.0, 1.0, 0.0]])  # one untouched dim, then the two pairs (1, 0), (1, 0)
    y = oracle.rope_partial(x, [100.0], rope_dims=4)
    c1, s1 = math.cos(1.0), math.sin(1.0)
    c100, s100 = math.cos(100.0), math.sin(100.0)
    assert np.allclose(y, [[9.0, c100, s100, c1, s1]], atol=1e-12)


def test_attention_sink_is_a_value_free_logit_in_the_softmax():
    # brute force over a tiny multiset: scores z with values v, plus the sink logit s
    # whose value is the zero vector, through numpy's softmax
    r = _rng(65)
    z, v = r.normal(size=(3, 2, 6)), r.normal(size=(3, 2, 6, 5))  # [rows][heads][entries](, dims)
    s = np.array([0.7, -1.2])
    o = np.einsum("rhe,rhed->rhd", np.exp(z - z.max(-1, keepdims=True)) /
                  np.exp(z - z.max(-1, keepdims=True)).sum(-1, keepdims=True), v)
    lse = np.log(np.exp(z).sum(-1))
    zs = np.concatenate([z, np.broadcast_to(s[None, :, None], (3, 2, 1))], axis=-1)
    p = np.exp(zs - zs.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    want = np.einsum("rhe,rhed->rhd", p[..., :6], v)  # the sink's value is zero
    out, l2 = oracle.sink_merge(o, lse, s)
    assert np.allclose(out, want, atol=1e-12)
    assert np.allclose(l2, np.log(np.exp(zs).sum(-1)), atol=1e-12)


def test_attention_sink_special_cases():
    r = _rng(66)
    o, lse = r.normal(size=(4, 3, 8)), r.normal(size=(4, 3))
    out, l2 = oracle.sink_merge(o, lse, np.full(3, -np.inf))  # no sink
    assert np.array_equal(out, o) and np.array_equal(l2, lse)
    out, l2 = oracle.sink_merge(o, lse, lse[0])  # row 0: the sink weighs as much as the branch
    assert np.allclose(out[0], o[0] / 2, atol=1e-12) and np.allclose(l2[0], lse[0] + math.log(2), atol=1e-12)
    out, l2 = oracle.sink_merge(o, np.full((4, 3), -np.inf), np.zeros(3))  # empty branch: zero output
    assert np.all(out == 0) and np.allclose(l2, 0.0)


# ------------------------------------------- grouped output projection ([HA] V.3)


def test_grouped_projection_is_a_block_diagonal_matmul():
    import scipy.linalg

    r = _rng(71)
    n_h, c, g, d_g = 8, 6, 4, 5
    o = r.normal(size=(3, 2, n_h, c))
    W = r.normal(size=(g, d_g, (n_h // g) * c))
    got = oracle.grouped_out_proj(o, W)
    want = o.reshape(3, 2, n_h * c) @ scipy.linalg.block_diag(*W).T
    assert got.shape == (3, 2, g * d_g) and np.allclose(got, want, atol=1e-12)


def test_grouped_projection_with_one_group_is_a_plain_projection_and_maps_to_d():
    r = _rng(72)
    n_h, c, d_g, d = 4, 3, 7, 5
    o = r.normal(size=(6, n_h, c))
    W = r.normal(size=(1, d_g, n_h * c))
    assert np.allclose(oracle.grouped_out_proj(o, W), o.reshape(6, -1) @ W[0].T, atol=1e-12)
    W_out = r.normal(size=(d, d_g))
    assert np.allclose(oracle.grouped_out_proj(o, W, W_out), o.reshape(6, -1) @ W[0].T @ W_out.T, atol=1e-12)


def test_grouped_projection_keeps_groups_apart():
    # a change in head h moves only the output block of its group h // (n_h / g)
    r = _rng(73)
    n_h, c, g, d_g = 8, 4, 4, 3
    o = r.normal(size=(1, n_h, c))
    W = r.normal(size=(g, d_g, (n_h // g) * c))
    base = oracle.grouped_out_proj(o, W)
    for h in range(n_h):
        o2 = o.copy()
        o2[0, h] += 1.0
        moved = np.abs(oracle.grouped_out_proj(o2, W) - base).reshape(g, d_g).max(axis=1) > 0
        assert np.array_equal(moved, np.arange(g) == h // (n_h // g))


# --------------------------------------------------- MXFP4 (indexer's FP4 path)


def test_e2m1_values_are_the_microscaling_grid():
    v = oracle.e2m1_decode(np.arange(16))
    # the eight magnitudes of e2m1 and their negatives (sign bit = bit 3)
    assert list(v[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(v[8:], -v[:8]) and math.copysign(1.0, v[8]) == -1.0


def test_e8m0_scales_are_powers_of_two():
    s = oracle.e8m0_decode(np.array([0, 1, 126, 127, 128, 254, 255]))
    assert list(s[:6]) == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127] and np.isnan(s[6])


def test_e2m1_encode_rounds_to_nearest_ties_to_even_and_saturates():
    grid = oracle.e2m1_decode(np.arange(8))
    assert np.array_equal(oracle.e2m1_encode(grid), np.arange(8))
    # midpoints: 0.25 -> 0 (code 0), 1.25 -> 1 (code 2), 2.5 -> 2 (code 4), 3.5 -> 4 (code 6), 5 -> 4 (code 6)
    assert list(oracle.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])) == [0, 2, 2, 4, 4, 6, 6]
    assert list(oracle.e2m1_encode([6.5, 100.0, -7.0])) == [7, 7, 15]
    assert list(oracle.e2m1_encode([-0.5, -0.0])) == [9, 8]


def test_mxfp4_worked_blocks():
    # amax 12: floor(log2 12) = 3, shared exponent 3 - 2 = 1, scale 2: 1, 2, 3, 12 land on the grid
    x = np.zeros((1, 64), dtype=np.float32)
    x[0, :4] = [1, 2, 3, 12]
    # second block: amax 7, shared exponent 0: 7 saturates to 6 (the format's clipping), 2.6 -> 3
    x[0, 32:35] = [7, 2.6, -0.2]
    codes, scales = oracle.quantise_mxfp4_rows(x)
    assert list(scales[0]) == [128, 127]
    y = oracle.mxfp4_decode(codes, scales)
    assert list(y[0, :4]) == [1.0, 2.0, 3.0, 12.0] and np.all(y[0, 4:32] == 0)
    assert list(y[0, 32:35]) == [6.0, 3.0, 0.0]
    z = oracle.quantise_mxfp4_rows(np.zeros((2, 32), dtype=np.float32))
    assert np.all(z[0] == 0) and np.all(z[1] == 0)  # all-zero block: smallest scale, zero codes


def test_mxfp4_error_is_within_half_a_grid_step():
    x = (_rng(74).normal(size=(50, 128)) * _rng(75).uniform(1e-3, 1e3, size=(50, 1))).astype(np.float32)
    codes, scales = oracle.quantise_mxfp4_rows(x)
    y = oracle.mxfp4_decode(codes, scales)
    s = np.repeat(oracle.e8m0_decode(scales), 32, axis=-1)
    u = np.abs(x) / s  # in units of the block's scale
    assert np.all(u.reshape(50, 4, 32).max(axis=-1) >= 4) and np.all(u < 8)  # normalisation of each block
    step = np.where(u < 2, 0.5, np.where(u < 4, 1.0, 2.0))  # grid spacing around |x| / scale
    bound = np.where(u <= 6, step / 2, u - 6) * s
    assert np.all(np.abs(y - x) <= bound + 1e-12)
