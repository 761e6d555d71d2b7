"""Host logic of the incremental decode session: ring slots and views (no GPU).

Every token's rows carry its position as their value, so a view of a ring can be
read back as the list of positions it holds.
"""
import torch

from sparse_attention_gated_b300.session import DecodeSession

B, C, CI, M, MH, W = 2, 8, 4, 4, 16, 8


def _session():
    return DecodeSession(batch=B, n_max=256, n_h=1, c=C, m=M, m_hca=MH, k=4, n_ih=1, c_I=CI, n_win=W,
                         bias=torch.zeros(2 * M, C), biasI=torch.zeros(2 * M, CI), bias_h=torch.zeros(MH, C),
                         device="cpu", dtype=torch.float32)


def _rows(p):
    r = {}
    for s in ("ca", "cb", "za", "zb", "ch", "zh", "kv", "kv_h"):
        r[s] = torch.full((B, C), float(p))
    for s in ("kIa", "kIb", "zIa", "zIb"):
        r[s] = torch.full((B, CI), float(p))
    return r


def _positions(view):
    """[B, rows, width] view of marker rows -> the positions of sequence 0 (all equal across b)."""
    assert torch.equal(view[0], view[-1])
    return [int(v) for v in view[0, :, 0].tolist()]


def _check_views(s, t):
    """What step t reads: the CSA block view when t completes a block, the HCA block,
    the window rows."""
    if (t + 1) % M == 0:
        i = (t + 1) // M - 1
        start, rows, fb, row0 = DecodeSession.csa_block_view(i, M)
        for name in ("ca", "zb", "kIa", "zIb"):
            got = _positions(s.ring(name)[:, start:start + rows])
            assert got == list(range(fb * M, fb * M + rows)), (t, name, got)
        # the call writes entries row0.. : the first one it produces (its first block
        # is only the previous block of the next when first_block > 0)
        assert row0 == (fb if fb == 0 else fb + 1)
    if (t + 1) % MH == 0:
        j = (t + 1) // MH - 1
        assert _positions(s.ring("ch")[:, :MH]) == list(range(j * MH, (j + 1) * MH))
    for name in ("kv", "kv_h"):
        kw, pos0 = s._window(name, t)
        n = min(W, t + 1)
        assert pos0 == max(0, t - W + 1)
        assert _positions(kw[:, :n]) == list(range(pos0, pos0 + n))


def test_rings_hold_what_each_step_reads():
    s = _session()
    for t in range(120):
        s.append(_rows(t))
        _check_views(s, t)
        s.t += 1


def test_prefill_rings_match_appending_token_by_token():
    for n0 in (0, 1, 3, 4, 5, 15, 16, 17, 31, 37, 64):
        a, b = _session(), _session()
        chunk = {k: torch.stack([_rows(p)[k] for p in range(n0)], dim=1) if n0 else torch.zeros(B, 0, v.shape[1])
                 for k, v in _rows(0).items()}
        a.fill_rings(chunk)
        for p in range(n0):
            b.append(_rows(p), p)
        b.t = n0
        assert a.t == n0
        # both continue the same way and read the same views
        for t in range(n0, n0 + 40):
            for s in (a, b):
                s.append(_rows(t))
                _check_views(s, t)
                s.t += 1


def test_window_view_stays_inside_its_allocation():
    s = _session()
    base = s.rings.data_ptr()
    end = base + s.rings.numel() * s.rings.element_size()
    for name in ("kv", "kv_h"):
        for t in range(3 * W):
            kw, _ = s._window(name, t)
            assert base <= kw.data_ptr() and kw.data_ptr() + kw.numel() * kw.element_size() <= end


def test_append_writes_every_slot_of_the_token_and_nothing_else():
    s = _session()
    for p in range(40):
        before = (s.rings.clone(), s.rings_I.clone())
        s.append(_rows(p + 1000), p)
        changed = (s.rings != before[0]).any(dim=-1).any(dim=1)  # [ring, row]
        changed_I = (s.rings_I != before[1]).any(dim=-1).any(dim=1)
        want = torch.zeros_like(changed)
        want_I = torch.zeros_like(changed_I)
        for name, views in s.token_slots(p).items():
            for v in views:
                assert torch.equal(v, torch.full_like(v, float(p + 1000)))
        for name in ("ca", "cb", "za", "zb", "ch", "zh", "kv", "kv_h"):
            r = ("ca", "cb", "za", "zb", "ch", "zh", "kv", "kv_h").index(name)
            for j in range(1 if name in ("ch", "zh") else 2):
                want[r, s._slot(name, j, p)] = True
        for r, name in enumerate(("kIa", "kIb", "zIa", "zIb")):
            for j in range(2):
                want_I[r, s._slot(name, j, p)] = True
        assert torch.equal(changed, want) and torch.equal(changed_I, want_I)
