"""The C ABI on the host: the library loads, exports what the header
declares, and validates/declines before touching any GPU."""

import ctypes
import os

import pytest

from dense_decoder_layer_gb300 import pds

pytestmark = pytest.mark.skipif(not os.path.exists(pds.LIB_PATH),
                                reason="libpds.so not built (run __graft_entry__.build())")


def _dims(**kw):
    base = dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=768,
                rope_theta=1.0e4, rms_eps=1e-5, rope_layout=0, rot_dim=0, freq_factors=None,
                rope_mscale=0.0, attn_softcap=0.0, window=0)
    base.update(kw)
    ff = base.pop("freq_factors")
    d = pds.pds_dims(*[base[f] for f, _ in pds.pds_dims._fields_ if f != "freq_factors"][:8])
    for f, _ in pds.pds_dims._fields_[8:]:
        if f == "freq_factors":
            if ff is not None:
                arr = (ctypes.c_float * len(ff))(*ff)
                d.freq_factors = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
                d._keep = arr
        else:
            setattr(d, f, base[f])
    return d


def _create(**kw):
    lib = pds.load()
    plan = ctypes.c_void_p()
    st = lib.pds_plan_create(ctypes.byref(_dims(**kw)), ctypes.byref(plan))
    return st, plan


def test_every_declared_function_is_exported():
    lib = pds.load()
    names = pds.header_functions()
    assert "pds_prefill_dense_stack" in names and "pds_plan_create" in names
    for n in names:
        assert hasattr(lib, n), n


def test_plan_create_accepts_the_served_shapes():
    for kw in ({}, dict(n_layers=16, d_model=2048, n_heads=32, n_kv_heads=8, ffn_dim=8192),
               dict(n_layers=28, d_model=3072, n_heads=24, n_kv_heads=8, head_dim=128,
                    ffn_dim=8192, rope_theta=5e5)):
        st, plan = _create(**kw)
        assert st == pds.PDS_OK, pds.last_error()
        assert pds.pds_workspace_bytes(plan, 512) > 0
        assert pds.pds_workspace_bytes(plan, 0) == 0
        # room for chunked attention grows with the prefix
        assert (pds.pds_workspace_bytes(plan, 512, 32768) > pds.pds_workspace_bytes(plan, 512, 0))
        pds.pds_plan_destroy(plan)


@pytest.mark.parametrize("kw", [dict(head_dim=96), dict(n_heads=5, n_kv_heads=2),
                                dict(d_model=200), dict(ffn_dim=700),
                                dict(n_heads=1, n_kv_heads=1, head_dim=64)])
def test_plan_create_declines_unserved_shapes(kw):
    st, plan = _create(**kw)
    assert st == pds.PDS_DECLINED
    assert not plan.value
    assert pds.last_error().startswith("declined")


@pytest.mark.parametrize("kw", [dict(n_layers=0), dict(d_model=-1), dict(rope_theta=0.0),
                                dict(rms_eps=-1.0), dict(rms_eps=float("nan"))])
def test_plan_create_rejects_bad_arguments(kw):
    st, _ = _create(**kw)
    assert st == pds.PDS_EINVAL


def test_null_arguments():
    lib = pds.load()
    assert lib.pds_plan_create(None, None) == pds.PDS_EINVAL
    lib.pds_plan_destroy(None)
    assert lib.pds_workspace_bytes(None, 8, 0) == 0
    assert lib.pds_workspace_bytes(None, 8, -1) == 0
    assert lib.pds_prefill_dense_stack(None, None, None, None, 0, 0, 1, None, None, None, 0,
                                       None) == pds.PDS_EINVAL


def test_disable_switch_declines(monkeypatch):
    monkeypatch.setenv("PDS_DISABLE", "1")
    st, _ = _create()
    assert st == pds.PDS_DECLINED
    monkeypatch.setenv("PDS_DISABLE", "0")
    st, plan = _create()
    assert st == pds.PDS_OK
    pds.pds_plan_destroy(plan)


def _fake_call(plan, cap, s, B, ws_bytes, device=True, layer_ptr=0x10000, ws=0x20000):
    """A call whose pointers are never dereferenced: it must be refused on the host."""
    L = 2
    layers = (pds.pds_layer * L)()
    for l in range(L):
        for f in pds.LAYER_FIELDS:
            setattr(layers[l], f, layer_ptr)
    kc = (ctypes.c_void_p * L)(*([0x30000] * L))
    vc = (ctypes.c_void_p * L)(*([0x40000] * L))
    fn = pds.load().pds_prefill_dense_stack_device if device else pds.load().pds_prefill_dense_stack
    return fn(plan, layers, kc, vc, cap, s, B, 0x50000, 0x60000, ws, ws_bytes, None)


def test_capacity_overflow_declines_before_any_device_work():
    st, plan = _create()
    ws = pds.pds_workspace_bytes(plan, 8)
    assert _fake_call(plan, cap=16, s=10, B=8, ws_bytes=ws) == pds.PDS_DECLINED
    assert _fake_call(plan, cap=16, s=10, B=8, ws_bytes=ws, device=False) == pds.PDS_DECLINED
    pds.pds_plan_destroy(plan)


def test_bad_calls_are_invalid():
    st, plan = _create()
    ws = pds.pds_workspace_bytes(plan, 8)
    assert _fake_call(plan, cap=16, s=0, B=0, ws_bytes=ws) == pds.PDS_EINVAL
    assert _fake_call(plan, cap=16, s=-1, B=8, ws_bytes=ws) == pds.PDS_EINVAL
    assert _fake_call(plan, cap=16, s=0, B=8, ws_bytes=ws - 1) == pds.PDS_EINVAL
    assert _fake_call(plan, cap=16, s=0, B=8, ws_bytes=ws, layer_ptr=0x10004) == pds.PDS_EINVAL
    assert _fake_call(plan, cap=16, s=0, B=8, ws_bytes=ws, ws=0x20008) == pds.PDS_EINVAL
    assert "16-byte" in pds.last_error()
    pds.pds_plan_destroy(plan)


def test_component_entry_points_validate_on_host():
    lib = pds.load()
    assert lib.pds_gemm_bf16(None, None, None, 8, 128, 64, None, 0, None) == pds.PDS_EINVAL
    assert lib.pds_gemm_bf16(0x100, 0x100, 0x100, 8, 100, 64, 0x100, 1 << 30, None) == pds.PDS_EINVAL
    assert lib.pds_gemm_bf16(0x100, 0x100, 0x100, 8, 192, 64, 0x100, 1 << 30, None) == pds.PDS_DECLINED
    assert lib.pds_gemm_bf16(0x100, 0x100, 0x100, 8, 256, 64, 0x100, 16, None) == pds.PDS_EINVAL
    assert pds.pds_gemm_workspace_bytes(512, 5120) >= pds.pds_gemm_workspace_bytes(8, 128) > 0
    assert lib.pds_attention(0x100, 0x100, 0x100, 0x100, 4, 0, 4, 2, 96, 0.0, 0, None, 0, None) == \
        pds.PDS_DECLINED
    assert lib.pds_attention(0x100, 0x100, 0x100, 0x100, 4, 0, 5, 2, 64, 0.0, 0, None, 0, None) == \
        pds.PDS_DECLINED
    assert lib.pds_attention(0x100, 0x100, 0x100, 0x100, 0, 0, 4, 2, 64, 0.0, 0, None, 0, None) == \
        pds.PDS_EINVAL


def test_stack_marshals_pointer_arrays_once():
    """DenseStack hands the C ABI pointer arrays built once (not per call);
    they hold exactly the tensors' addresses, and the marshalling helpers pass
    such arrays through unchanged."""
    torch = pytest.importorskip("torch")
    import synth
    from dense_decoder_layer_gb300.stack import DenseStack
    dims = synth.CONFIGS["tiny"]
    st = DenseStack(dims, 32, 8, device="cpu")
    try:
        assert [st._k_ptrs[i] for i in range(dims.n_layers)] == \
            [t.data_ptr() for t in st.k_cache]
        assert [st._v_ptrs[i] for i in range(dims.n_layers)] == \
            [t.data_ptr() for t in st.v_cache]
        layers = [{n: torch.empty(16, dtype=torch.bfloat16) for n in pds.LAYER_FIELDS}
                  for _ in range(dims.n_layers)]
        st.set_layer_tensors(layers)
        for l, arr in zip(layers, st._layers_c):
            for n in pds.LAYER_FIELDS:
                assert getattr(arr, n) == l[n].data_ptr()
        assert pds._ptrs(st._k_ptrs) is st._k_ptrs
        assert pds._layer_array(st._layers_c) is st._layers_c
    finally:
        st.close()


@pytest.mark.parametrize("kw", [dict(rope_layout=1), dict(rot_dim=32), dict(rot_dim=64),
                                dict(rope_layout=1, rot_dim=16),
                                dict(freq_factors=[1.0 + i for i in range(32)]),
                                dict(rope_mscale=1.2, attn_softcap=30.0, window=128)])
def test_plan_create_accepts_the_served_variants(kw):
    st, plan = _create(**kw)
    assert st == pds.PDS_OK, pds.last_error()
    pds.pds_plan_destroy(plan)


@pytest.mark.parametrize("kw", [dict(rot_dim=16), dict(rot_dim=48), dict(rope_layout=1, rot_dim=8)])
def test_plan_create_declines_unserved_rotary_widths(kw):
    st, plan = _create(**kw)
    assert st == pds.PDS_DECLINED, pds.last_error()
    assert not plan.value


@pytest.mark.parametrize("kw", [dict(rope_layout=2), dict(rot_dim=-2), dict(rot_dim=66),
                                dict(rot_dim=3), dict(rope_mscale=-1.0),
                                dict(attn_softcap=-1.0), dict(attn_softcap=float("inf")),
                                dict(window=-1), dict(freq_factors=[1.0] * 31 + [0.0]),
                                dict(freq_factors=[1.0] * 31 + [float("nan")])])
def test_plan_create_rejects_bad_variants(kw):
    st, _ = _create(**kw)
    assert st == pds.PDS_EINVAL, pds.last_error()


def test_attention_entry_rejects_negative_options():
    lib = pds.load()
    args = (0x100, 0x100, 0x100, 0x100, 8, 0, 4, 2, 64)
    assert lib.pds_attention(*args, -1.0, 0, None, 0, None) == pds.PDS_EINVAL
    assert lib.pds_attention(*args, 0.0, -5, None, 0, None) == pds.PDS_EINVAL


def test_plan_without_a_device_is_host_only():
    """On a machine without a CUDA device the plan still validates and sizes
    its workspace; a call then fails after admission instead of touching a GPU."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    st, plan = _create()
    assert st == pds.PDS_OK
    L = 2
    layers = (pds.pds_layer * L)()
    for l in range(L):
        for f in pds.LAYER_FIELDS:
            setattr(layers[l], f, 0x10000)
    kc = (ctypes.c_void_p * L)(*([0x30000] * L))
    vc = (ctypes.c_void_p * L)(*([0x40000] * L))
    ws = pds.pds_workspace_bytes(plan, 8)
    rc = pds.load().pds_prefill_dense_stack_device(plan, layers, kc, vc, 16, 0, 8, 0x50000,
                                                   0x60000, 0x20000, ws, None)
    assert rc == pds.PDS_ELAUNCH
    assert "without a CUDA device" in pds.last_error()
    pds.pds_plan_destroy(plan)


def test_attention_workspace_sizes():
    assert pds.pds_attention_workspace_bytes(512, 0, 24, 128) < \
        pds.pds_attention_workspace_bytes(512, 32768, 24, 128)
    assert pds.pds_attention_workspace_bytes(0, 0, 24, 128) == 0
    assert pds.pds_attention_workspace_bytes(8, 0, 24, 96) == 0
