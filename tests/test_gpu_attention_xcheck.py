"""The tcgen05 attention kernel against the warp-level mma.sync kernel of the
test-only library (tests/xcheck): two independent GPU implementations of the
same attention, on the same inputs."""

import ctypes
import os

import pytest

from parity import assert_parity, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

XCHECK_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "xcheck",
                          "libpds_xcheck.so")


def _xcheck():
    lib = ctypes.CDLL(XCHECK_LIB)
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.pdsx_attention_mma.restype = ctypes.c_int
    lib.pdsx_attention_mma.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    return lib


@pytest.mark.parametrize("shape", [(512, 1536, 24, 8, 128), (300, 77, 8, 2, 64)])
def test_tcgen05_attention_matches_mma_kernel(shape):
    from dense_decoder_layer_gb300 import pds
    B, s, H, Hkv, hd = shape
    g = torch.Generator().manual_seed(B + s)
    q = torch.randn(B, H, hd, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(s + B, Hkv, hd, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(s + B, Hkv, hd, generator=g).to(torch.bfloat16).cuda()
    o_tc = torch.empty(B, H * hd, dtype=torch.bfloat16, device="cuda")
    o_mma = torch.empty_like(o_tc)
    stream = torch.cuda.current_stream().cuda_stream
    pds.pds_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_tc.data_ptr(), B, s, H, Hkv,
                      hd, stream)
    assert _xcheck().pdsx_attention_mma(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        o_mma.data_ptr(), B, s, H, Hkv, hd, stream) == 0
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    assert_parity(bf16_to_f64(o_tc), bf16_to_f64(o_mma), f"tcgen05 vs mma.sync attention {shape}")
