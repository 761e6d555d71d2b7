"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/hyb.h declares, and rejects invalid arguments before any
launch."""
import ctypes
import os
import re

import pytest
import torch

from sparse_attention_gated_b300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "hyb.h")).read()
    return set(re.findall(r"HYB_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        from sparse_attention_gated_b300 import build

        build.build()
    return _abi.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_abi.SIGNATURES) == declared


def test_library_reports_its_build(lib):
    assert lib.hyb_version() >= 1
    assert lib.hyb_built_arch() == 1030
    assert lib.hyb_status_string(0) == b"HYB_OK"


def test_out_count_matches_the_append_rule(lib):
    assert lib.hyb_compress_out_count(16, 4, 1, 0) == 4
    assert lib.hyb_compress_out_count(8, 4, 1, 5) == 1
    assert lib.hyb_compress_out_count(8, 4, 1, 0) == 2
    assert lib.hyb_compress_out_count(255, 4, 0, 0) == 63
    assert lib.hyb_compress_out_count(3, 4, 1, 0) == 0


FAKE = 1 << 20  # a well-aligned non-null address; validation fails before anything is launched


def _compress_args(**kw):
    a = _abi.CompressArgs()
    a.ca = a.za = a.bias = a.out = FAKE
    a.cb = a.zb = FAKE
    a.batch, a.n_rows, a.c, a.m, a.overlap = 1, 16, 64, 4, 1
    a.in_dtype, a.out_dtype = _abi.HYB_F32, _abi.HYB_F32
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,status", [
    (dict(ca=None), 1), (dict(m=0), 1), (dict(overlap=2), 1), (dict(in_dtype=_abi.HYB_E4M3), 1),
    (dict(c=48), 2), (dict(out_dtype=_abi.HYB_E4M3), 1), (dict(ca=FAKE + 4), 1), (dict(zb=None), 1),
    (dict(out_batch_stride=2), 1), (dict(batch=-1), 1), (dict(in_batch_stride=8), 1), (dict(in_batch_stride=-1), 1),
])
def test_compress_rejects_invalid_arguments(lib, change, status):
    a = _compress_args(**change)
    assert lib.hyb_compress(ctypes.byref(a), None, 0, None) == status
    assert lib.hyb_last_error()


def test_compress_with_nothing_to_do_launches_nothing(lib):
    a = _compress_args(n_rows=3)
    assert lib.hyb_compress(ctypes.byref(a), None, 0, None) == 0


def test_compress_batch_validates_every_call_before_any_launch(lib):
    arr = (_abi.CompressArgs * 5)(*[_compress_args(n_rows=3) for _ in range(5)])  # nothing to compute
    assert lib.hyb_compress_batch(arr, 0, None) == 0
    assert lib.hyb_compress_batch(arr, 4, None) == 0
    assert lib.hyb_compress_batch(arr, 5, None) == 1  # more than HYB_COMPRESS_BATCH_MAX calls
    assert lib.hyb_compress_batch(arr, -1, None) == 1
    assert lib.hyb_compress_batch(None, 2, None) == 1
    bad = (_abi.CompressArgs * 3)(_compress_args(n_rows=3), _compress_args(n_rows=3, m=0), _compress_args(n_rows=3))
    assert lib.hyb_compress_batch(bad, 3, None) == 1  # the second call is invalid
    mixed = (_abi.CompressArgs * 2)(_compress_args(n_rows=3), _compress_args(n_rows=3, in_dtype=_abi.HYB_BF16))
    assert lib.hyb_compress_batch(mixed, 2, None) == 1
    assert "in_dtype" in lib.hyb_last_error().decode()


def test_mxfp4_arguments_are_validated_before_any_launch(lib):
    # compression to MXFP4 needs the scale bytes (and only scaled outputs take them)
    assert lib.hyb_compress(ctypes.byref(_compress_args(c=128, out_dtype=_abi.HYB_MXFP4)), None, 0, None) == 1
    assert lib.hyb_compress(ctypes.byref(_compress_args(c=48, out_dtype=_abi.HYB_MXFP4, out_scale=FAKE)), None, 0,
                            None) == 2  # (c not compiled)
    # the MXFP4 indexer runs on the tensor cores only: 64 heads x 128 dims
    a = _index_args(dtype=_abi.HYB_MXFP4, qI_scale=FAKE, kI_scale=FAKE)  # 4 heads x 32 dims
    assert lib.csa_index_topk(ctypes.byref(a), None, 0, None) == 2
    assert "MXFP4" in lib.hyb_last_error().decode()
    a = _index_args(dtype=_abi.HYB_MXFP4)  # no scales
    assert lib.csa_index_topk(ctypes.byref(a), None, 0, None) == 1


def test_binding_maps_the_fp4_formats():
    from sparse_attention_gated_b300 import ops

    assert ops._DT[torch.float4_e2m1fn_x2] == _abi.HYB_MXFP4


def _index_args(**kw):
    a = _abi.IndexArgs()
    a.qI = a.w = a.kI = a.idx = FAKE
    a.batch, a.n_q, a.n_entries, a.n_ih, a.c_I, a.m, a.k, a.q_pos0 = 1, 4, 100, 4, 32, 4, 16, 0
    a.dtype = _abi.HYB_F32
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,status", [
    (dict(qI=None), 1), (dict(k=0), 1), (dict(k=4096), 2), (dict(dtype=_abi.HYB_BF16), 1),
    (dict(q_pos0=1000), 1), (dict(c_I=24), 2), (dict(dtype=_abi.HYB_E4M3), 1), (dict(qI_scale=FAKE), 1),
    (dict(kI=FAKE + 8), 1), (dict(kv_stride=50), 1),
])
def test_index_rejects_invalid_arguments(lib, change, status):
    a = _index_args(**change)
    assert lib.csa_index_topk(ctypes.byref(a), FAKE, 1 << 30, None) == status


def test_index_requires_a_workspace(lib):
    a = _index_args()
    assert lib.csa_index_topk_workspace_size(ctypes.byref(a)) > 0
    assert lib.csa_index_topk(ctypes.byref(a), None, 0, None) == 3


def test_attend_and_merge_reject_invalid_arguments(lib):
    a = _abi.CsaAttendArgs()
    a.q = a.kc = a.vc = a.idx = a.o = a.lse = FAKE
    a.batch, a.n_q, a.n_h, a.c, a.n_entries, a.k, a.scale, a.dtype = 1, 2, 4, 64, 10, 4, 0.1, _abi.HYB_E4M3
    assert lib.csa_attend(ctypes.byref(a), None, 0, None) == 1
    a.dtype = _abi.HYB_F32
    a.c = 96
    assert lib.csa_attend(ctypes.byref(a), None, 0, None) == 2
    a.c = 64
    a.sink = FAKE + 2  # sink logits must be float-aligned
    assert lib.csa_attend(ctypes.byref(a), None, 0, None) == 1
    assert "sink" in lib.hyb_last_error().decode()
    a.sink = None
    h = _abi.HcaAttendArgs()
    h.q = h.kc = h.vc = h.o = h.lse = FAKE
    h.batch, h.n_q, h.n_h, h.c, h.n_entries, h.m, h.q_pos0, h.dtype = 1, 1, 4, 64, 3, 16, 100, _abi.HYB_F32
    assert lib.hca_attend(ctypes.byref(h), None, 0, None) == 1  # position 100 sees 6 entries, only 3 exist
    s = _abi.SwaArgs()
    s.q = s.kw = s.vw = s.out = FAKE
    s.batch, s.n_q, s.n_h, s.c, s.n_kv, s.kv_pos0, s.q_pos0, s.n_win = 1, 1, 4, 64, 16, 100, 200, 16
    s.dtype = s.out_dtype = _abi.HYB_F32
    assert lib.swa_merge(ctypes.byref(s), None, 0, None) == 1  # window rows outside the buffer
    s.kv_pos0, s.o_in = 185, FAKE
    assert lib.swa_merge(ctypes.byref(s), None, 0, None) == 1  # o_in without lse_in


def test_noalloc_indexer_rejects_sizes_beyond_its_scratch(lib):
    """The allocation-free indexer needs csa_index_topk's workspace to fit its fixed
    scratch; larger problems are rejected on the host, before any CUDA call."""
    a = _abi.IndexArgs()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call is rejected first
    a.qI = a.qI_scale = a.w = a.kI = a.kI_scale = a.idx = fake
    a.batch, a.n_q, a.n_entries, a.kv_stride, a.n_ih, a.c_I, a.m, a.k = 64, 1, 1 << 20, 1 << 20, 64, 128, 4, 1024
    a.q_pos0 = 4 * (1 << 20) - 1
    a.dtype = _abi.HYB_E4M3
    need = lib.csa_index_topk_workspace_size(ctypes.byref(a))
    assert need > _abi.HYB_NOALLOC_SCRATCH_BYTES
    assert lib.csa_index_topk_noalloc(ctypes.byref(a), None) == 3  # HYB_ERR_WORKSPACE
    assert b"scratch" in lib.hyb_last_error()


def test_packed_step_io_keeps_values_and_aliases_one_buffer():
    """HybridStep.pack_step_io: every per-step input (and output) becomes a view of one
    contiguous buffer at a 256-byte aligned offset, with its values unchanged."""
    from sparse_attention_gated_b300 import pipeline, workloads

    w = workloads.scaled(workloads.WORKLOADS["tiny_f32"], n_ctx=64)
    # the buffers only (constructing a step sizes workspaces through the CUDA library)
    st = pipeline.HybridStep.__new__(pipeline.HybridStep)
    st.w, st.x, st.device = w, workloads.make_inputs(w, device="cpu"), torch.device("cpu")
    st.buf = {"out": torch.randn(1, 64, 4, 64), "out_h": torch.randn(1, 64, 4, 64)}
    before = {k: st.x[k].clone() for k in st.step_input_keys()}
    outs_before = {k: st.buf[k].clone() for k in st.output_keys()}
    dev_in, dev_out = st.pack_step_io()
    base = dev_in.data_ptr()
    for k, v in before.items():
        t = st.x[k]
        assert torch.equal(t, v), k
        off = t.data_ptr() - base
        assert 0 <= off and off + t.numel() * t.element_size() <= dev_in.numel() and off % 256 == 0, k
    for k in st.output_keys():
        off = st.buf[k].data_ptr() - dev_out.data_ptr()
        assert 0 <= off < dev_out.numel() and off % 256 == 0, k
        assert torch.equal(st.buf[k], outs_before[k]), k


def test_rmsnorm_rope_rejects_invalid_arguments(lib):
    def args(**kw):
        a = _abi.NormRopeArgs()
        a.x, a.rows, a.c, a.eps, a.dtype = FAKE, 4, 64, 1e-6, _abi.HYB_F32
        a.pos, a.rows_per_pos, a.rope_dims, a.theta = FAKE, 1, 16, 10000.0
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    for bad in (dict(c=63), dict(c=0), dict(dtype=_abi.HYB_E4M3), dict(rope_dims=66), dict(rope_dims=15),
                dict(pos=None), dict(rows_per_pos=0), dict(theta=0.0), dict(eps=-1.0), dict(x=None), dict(x=FAKE + 4),
                dict(pos=FAKE + 4), dict(rows=-1), dict(row_stride=62), dict(row_stride=65)):
        assert lib.hyb_rmsnorm_rope(ctypes.byref(args(**bad)), None) == 1, bad
        assert lib.hyb_last_error()
    assert lib.hyb_rmsnorm_rope(ctypes.byref(args(rows=0)), None) == 0  # nothing to do, nothing launched


def test_rmsnorm_rope_batch_validates_every_call_before_any_launch(lib):
    def args(**kw):
        a = _abi.NormRopeArgs()
        a.x, a.rows, a.c, a.eps, a.dtype = FAKE, 4, 64, 1e-6, _abi.HYB_F32
        a.pos, a.rows_per_pos, a.rope_dims, a.theta = FAKE, 1, 16, 10000.0
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    def call(*calls, n=None):
        arr = (_abi.NormRopeArgs * max(1, len(calls)))(*calls)
        return lib.hyb_rmsnorm_rope_batch(arr, len(calls) if n is None else n, None)
    assert call(n=0) == 0  # nothing to do
    assert call(args(), n=5) == 1 and call(args(), n=-1) == 1
    assert call(args(), args(c=63)) == 1  # an invalid member
    assert call(args(), args(dtype=_abi.HYB_BF16)) == 1  # mixed dtypes
    assert call(args(rows=0), args(rows=0)) == 0  # nothing launched
    assert lib.hyb_rmsnorm_rope_batch(None, 1, None) == 1


def test_binding_rejects_bad_sink_positions_and_gain_before_any_call():
    from sparse_attention_gated_b300 import ops
    q = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        ops.csa_attend_args(q, q, q, None, 0.1, None, None, sink=torch.zeros(3))
    with pytest.raises(ValueError):
        ops.hca_attend_args(q, q, q, 4, 0, 0.1, None, None, sink=torch.zeros(4, dtype=torch.float64))
    x = torch.zeros(6, 64)
    with pytest.raises(ValueError):
        ops.rmsnorm_rope(x, pos=torch.zeros(5, dtype=torch.int64))  # 6 rows need 6 positions
    with pytest.raises(ValueError):
        ops.rmsnorm_rope(torch.zeros(2, 6, 64)[:, 1:4])  # neither contiguous nor 2-D rows
    with pytest.raises(ValueError):
        ops.rmsnorm_rope(torch.zeros(64, 6).t())  # columns not unit-stride
    with pytest.raises(ValueError):
        ops.rmsnorm_rope(x, pos=torch.zeros(6, dtype=torch.int32))
    with pytest.raises(ValueError):
        ops.rmsnorm_rope(x, gamma=torch.ones(32), pos=None)


def test_fused_window_arguments_are_validated_before_any_launch(lib):
    def csa(**w):
        win = _abi.Window()
        win.kw, win.out, win.out_dtype = FAKE, FAKE, _abi.HYB_BF16
        win.n_kv, win.kv_pos0, win.q_pos0, win.n_win = 256, 1000, 1127, 128
        for k, v in w.items():
            setattr(win, k, v)
        a = _abi.CsaAttendArgs()
        a.q = a.kc = a.vc = a.idx = a.lse = FAKE
        a.batch, a.n_q, a.n_h, a.c, a.n_entries, a.k, a.scale, a.dtype = 1, 1, 64, 512, 100, 16, 0.1, _abi.HYB_BF16
        a._w = win
        a.window = ctypes.cast(ctypes.pointer(win), ctypes.c_void_p)
        return a
    for bad in (dict(n_win=0), dict(out_dtype=_abi.HYB_E4M3), dict(kv_pos0=1001),  # first window row not held
                dict(n_kv=127), dict(q_pos0=-1), dict(kw=None), dict(out=None), dict(kw=FAKE + 2)):
        assert lib.csa_attend(ctypes.byref(csa(**bad)), None, 0, None) == 1, bad
        assert lib.hyb_last_error()
    h = _abi.HcaAttendArgs()
    h.q = h.kc = h.vc = h.lse = FAKE
    h.batch, h.n_q, h.n_h, h.c, h.n_entries, h.m, h.q_pos0, h.dtype = 1, 1, 64, 512, 100, 16, 1599, _abi.HYB_BF16
    win = _abi.Window()
    win.kw, win.out, win.out_dtype, win.n_kv, win.kv_pos0, win.q_pos0, win.n_win = FAKE, FAKE, _abi.HYB_BF16, 128, \
        1472, 1598, 128
    h.window = ctypes.cast(ctypes.pointer(win), ctypes.c_void_p)
    assert lib.hca_attend(ctypes.byref(h), None, 0, None) == 1  # the window's query is not the call's
    assert "q_pos0" in lib.hyb_last_error().decode()


def test_per_query_positions_are_checked_where_the_host_can(lib):
    """Per-query positions live in device memory: the host checks their pointers
    (8-byte alignment) and that a fused HCA window uses the call's own positions;
    the positions themselves are range-checked by the kernels."""
    a = _abi.IndexArgs()
    a.qI = a.w = a.kI = a.idx = FAKE
    a.batch, a.n_q, a.n_entries, a.n_ih, a.c_I, a.m, a.k, a.dtype = 2, 1, 1000, 8, 64, 4, 16, _abi.HYB_F32
    a.q_pos0 = 10 ** 9  # ignored with per-query positions (would see more entries than exist)
    a.q_pos = FAKE + 4
    assert lib.csa_index_topk(ctypes.byref(a), None, 0, None) == 1
    assert "q_pos" in lib.hyb_last_error().decode()
    a.q_pos = FAKE
    # sized for every row seeing all 1000 entries
    assert lib.csa_index_topk_workspace_size(ctypes.byref(a)) >= 2 * 1000 * 4
    assert lib.csa_index_topk(ctypes.byref(a), None, 0, None) == 3  # HYB_ERR_WORKSPACE: it got past validation
    h = _abi.HcaAttendArgs()
    h.q = h.kc = h.vc = h.lse = FAKE
    h.batch, h.n_q, h.n_h, h.c, h.n_entries, h.m, h.q_pos0, h.dtype = 1, 1, 64, 512, 100, 16, 0, _abi.HYB_BF16
    h.q_pos = FAKE + 8
    win = _abi.Window()
    win.kw, win.out, win.out_dtype, win.n_kv, win.kv_pos0, win.n_win = FAKE, FAKE, _abi.HYB_BF16, 128, 0, 128
    h.window = ctypes.cast(ctypes.pointer(win), ctypes.c_void_p)
    assert lib.hca_attend(ctypes.byref(h), None, 0, None) == 1  # the window has no per-query positions
    win.q_pos = FAKE + 8
    win.kv_pos0s = FAKE + 4
    assert lib.hca_attend(ctypes.byref(h), None, 0, None) == 1  # misaligned kv_pos0s
    win.kv_pos0s = FAKE
    assert lib.hca_attend(ctypes.byref(h), None, 0, None) == 3  # past validation: the workspace is missing
    s = _abi.SwaArgs()
    s.q = s.kw = s.vw = s.out = FAKE
    s.batch, s.n_q, s.n_h, s.c, s.n_kv, s.n_win, s.dtype, s.out_dtype = 1, 1, 64, 512, 10, 128, 1, 1
    s.q_pos0, s.kv_pos0 = 5000, 0  # rows outside the buffer: rejected as numbers ...
    assert lib.swa_merge(ctypes.byref(s), None, 0, None) == 1
    s.q_pos = FAKE  # ... not checkable as device-side positions (the kernel clips and reports)
    s.kv_pos0s = FAKE + 2
    assert lib.swa_merge(ctypes.byref(s), None, 0, None) == 1
