"""The no-allocation GEMM entry point (pds_gemm_bf16_noalloc).

It serves callers that cannot call cudaMalloc (a process whose device
memory is all held by its own pool, a plugin inside an application that
owns every allocation): its scratch is a static array in the library, not
a caller buffer.  Its result must match pds_gemm_bf16's, call after call,
although every call reuses the same static scratch.  This file is named to
be collected last.
"""

import ctypes
import os

import numpy as np
import pytest

import synth
from dense_decoder_layer_gb300 import pds
from parity import assert_parity


def _bf16(torch, rng, *shape, scale=1.0):
    bits = synth.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(512, 3072, 3072), (130, 384, 8192)])
def test_noalloc_gemm_matches_gemm_bf16_twice(M, N, K):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(M + N + K)
    a = _bf16(torch, rng, M, K)
    w = _bf16(torch, rng, N, K, scale=1 / np.sqrt(K))
    stream = torch.cuda.current_stream().cuda_stream
    ws_bytes = pds.pds_gemm_workspace_bytes(M, N)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    pds.pds_gemm_bf16(a.data_ptr(), w.data_ptr(), ref.data_ptr(), M, N, K, ws.data_ptr(),
                      ws_bytes, stream)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()
    for call in range(2):  # the second call finds the first call's leftovers in the scratch
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        pds.pds_gemm_bf16_noalloc(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, stream)
        # no bounded wait of the call gave up (the status word in the static scratch)
        assert pds.pds_component_sync(stream) == pds.PDS_OK
        assert_parity(c.cpu().numpy(), want, f"noalloc call {call} {M}x{N}x{K}", rel_l2=1e-5,
                      max_abs_rms=1e-4)


@pytest.mark.skipif(not os.path.exists(pds.LIB_PATH), reason="libpds.so not built")
def test_noalloc_gemm_rejects_sizes_beyond_its_scratch():
    lib = pds.load()
    # 129 row tiles x 128 column tiles = 16512 > 16384 output tiles: refused on the host
    st = lib.pds_gemm_bf16_noalloc(0x100, 0x100, 0x100, 129 * 128, 128 * 128, 64, None)
    assert st == pds.PDS_EINVAL
    assert "static scratch" in pds.last_error()
    assert lib.pds_gemm_bf16_noalloc(0x100, 0x100, 0x100, 8, 192, 64, None) == pds.PDS_DECLINED
    assert "pds_gemm_bf16_noalloc" in pds.header_functions()
