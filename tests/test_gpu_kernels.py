"""Kernel-level parity through the C ABI's component entry points."""

import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _bf16(rng, *shape, scale=1.0):
    bits = synth.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t, synth.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(8, 256, 64), (1, 128, 64), (130, 384, 320), (128, 512, 4096),
                                   (200, 640, 8192), (512, 5120, 3072), (2048, 3072, 2048),
                                   (37, 128, 192),
                                   # one row tile over a cluster of c CTAs that finish row
                                   # slices: c = 4 with a ragged last slice, c = 4 with three or
                                   # two empty slices, c = 3 (48-row slices), c = 8 (16-row
                                   # slices, 128-wide tiles), c = 6 (24-row slices)
                                   (100, 768, 1024), (17, 128, 512), (64, 384, 512),
                                   (9, 256, 384), (120, 384, 1024), (128, 640, 768)])
def test_gemm_bf16_matches_fp64(M, N, K):
    from dense_decoder_layer_gb300 import pds
    rng = np.random.default_rng(M * 7 + N + K)
    a, a64 = _bf16(rng, M, K)
    w, w64 = _bf16(rng, N, K, scale=1 / np.sqrt(K))
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = pds.pds_gemm_workspace_bytes(M, N)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # second call reuses the scratch (counters must be back at zero)
        stream = torch.cuda.current_stream().cuda_stream
        pds.pds_gemm_bf16(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, ws.data_ptr(),
                          ws_bytes, stream)
        assert pds.pds_component_sync(stream) == pds.PDS_OK
        want = a64 @ w64.T
        assert_parity(c.cpu().numpy(), want, f"gemm {M}x{N}x{K}", rel_l2=1e-5, max_abs_rms=1e-4)


@pytest.mark.parametrize("B,s,H,Hkv,hd", [(1, 0, 4, 2, 64), (7, 0, 4, 2, 64), (130, 0, 8, 2, 64),
                                          (64, 100, 6, 2, 128), (200, 333, 3, 1, 128),
                                          (1, 77, 8, 8, 128), (512, 1536, 24, 8, 128),
                                          (129, 0, 32, 8, 64),
                                          # key ranges of 9-11 tiles, split over CTA pairs
                                          (300, 1000, 4, 2, 64), (130, 900, 5, 1, 128)])
def test_attention_matches_oracle(B, s, H, Hkv, hd):
    from dense_decoder_layer_gb300 import pds
    rng = np.random.default_rng(B + 11 * s + H)
    q, q64 = _bf16(rng, B, H, hd)
    k, k64 = _bf16(rng, s + B, Hkv, hd)
    v, v64 = _bf16(rng, s + B, Hkv, hd)
    o = torch.full((B, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    pds.pds_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, s, H, Hkv, hd,
                      stream)
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    want = oracle.causal_gqa_attention(q64, k64, v64, s).reshape(B, H * hd)
    assert_parity(bf16_to_f64(o), want, f"attention B={B} s={s} H={H}/{Hkv} hd={hd}")
