"""Failure detection: declines before device work, a failure after
admission reported once per distinct message, and device waits that give
up with a status instead of hanging.  Nothing here faults a GPU."""

import ctypes
import os

import pytest

from dense_decoder_layer_gb300 import pds

needs_lib = pytest.mark.skipif(not os.path.exists(pds.LIB_PATH), reason="libpds.so not built")


def _plan():
    dims = pds.pds_dims(2, 256, 4, 2, 64, 768, 1.0e4, 1e-5)
    return pds.pds_plan_create(dims)


def _fake_device_call(plan):
    L = 2
    layers = (pds.pds_layer * L)()
    for l in range(L):
        for f in pds.LAYER_FIELDS:
            setattr(layers[l], f, 0x10000)
    kc = (ctypes.c_void_p * L)(*([0x30000] * L))
    vc = (ctypes.c_void_p * L)(*([0x40000] * L))
    ws = pds.pds_workspace_bytes(plan, 8)
    return pds.load().pds_prefill_dense_stack_device(plan, layers, kc, vc, 16, 0, 8, 0x50000,
                                                     0x60000, 0x20000, ws, None)


@needs_lib
def test_injected_failure_after_admission_is_reported_once(monkeypatch, capfd):
    plan = _plan()
    monkeypatch.setenv("PDS_FAULT_AFTER_ADMIT", "1")
    for _ in range(3):
        assert _fake_device_call(plan) == pds.PDS_ELAUNCH
        assert "injected failure after admission" in pds.last_error()
    err = capfd.readouterr().err
    assert err.count("injected failure after admission") == 1
    monkeypatch.setenv("PDS_FAULT_AFTER_ADMIT", "0")
    pds.pds_plan_destroy(plan)


@needs_lib
def test_selftest_rejects_bad_limits():
    assert pds.load().pds_selftest_stuck_wait(0, None) == pds.PDS_EINVAL
    assert pds.load().pds_selftest_stuck_wait(20_000_000, None) == pds.PDS_EINVAL


@pytest.mark.gpu
def test_stuck_device_wait_times_out_and_gpu_stays_usable():
    """The component path reports a bounded wait that gave up, clears it, and
    the context stays usable: a GEMM right after runs and is right."""
    torch = pytest.importorskip("torch")
    stream = torch.cuda.current_stream().cuda_stream
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    pds.pds_selftest_stuck_wait(2000, stream)
    assert pds.pds_component_sync(stream) == pds.PDS_ETIMEOUT
    assert "gave up" in pds.last_error()
    assert pds.pds_component_sync(stream) == pds.PDS_OK  # read and cleared
    a = torch.randn(130, 128, device="cuda").to(torch.bfloat16)
    w = torch.randn(256, 128, device="cuda").to(torch.bfloat16)
    c = torch.empty(130, 256, device="cuda")
    wsb = pds.pds_gemm_workspace_bytes(130, 256)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    pds.pds_gemm_bf16(a.data_ptr(), w.data_ptr(), c.data_ptr(), 130, 256, 128, ws.data_ptr(), wsb,
                      stream)
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    ref = a.float() @ w.float().T
    assert float((c - ref).norm() / ref.norm()) < 1e-5
