"""Decode steps (B = 1 ... 8 new rows against a resident cache) and long
cached prefixes (8k and 32k rows) against the oracle, through the C ABI."""

import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, bf16_to_f64, oracle_result, run_gpu, run_oracle, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# The Llama-3.2-3B layer shape, a few layers, over a 2048-row cache.
DEC = synth.Dims(3, 3072, 24, 8, 128, 8192, 8, 2048, 5.0e5)


def _check(got, want, tag):
    assert_parity(got[0], want[0], f"{tag} hidden_out")
    for l in range(len(want[1])):
        assert_parity(got[1][l], want[1][l], f"{tag} k_rows[{l}]")
        assert_parity(got[2][l], want[2][l], f"{tag} v_rows[{l}]")


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8])
def test_decode_step_matches_oracle(B):
    dims = DEC.replace(batch=B)
    dims, (layers, pk, pv, hidden) = workload(dims)
    _check(run_gpu(dims, layers, pk, pv, hidden), oracle_result(dims), f"decode B={B}")


def test_prefill_then_decode_steps_match_one_prefill():
    """A 100-row prefill over a 300-row prefix, then decode steps of 1, 2, 5
    and 8 rows, each appending to the caches: every step's output and K/V
    rows equal the oracle's single prefill of all 116 rows."""
    from dense_decoder_layer_gb300.stack import DenseStack
    steps = [100, 1, 2, 5, 8]
    total = sum(steps)
    dims = synth.Dims(2, 1024, 8, 2, 128, 2048, total, 300, 5.0e5)
    dims, (layers, pk, pv, hidden) = workload(dims)
    want = run_oracle(dims, layers, pk, pv, hidden)
    st = DenseStack(dims, dims.start_pos + total, max(steps))
    st.load_layers(layers)
    st.load_prefix(pk, pv)
    b = 0
    for n in steps:
        out = st.prefill(torch.from_numpy(hidden[b:b + n].copy()), dims.start_pos + b).numpy()
        assert_parity(out.astype(np.float64), want[0][b:b + n], f"step of {n} at row {b}")
        for l in range(dims.n_layers):
            k, v = st.rows(l, dims.start_pos + b, n)
            assert_parity(bf16_to_f64(k), want[1][l][b:b + n], f"step {n} k[{l}]")
            assert_parity(bf16_to_f64(v), want[2][l][b:b + n], f"step {n} v[{l}]")
        b += n
    st.close()


def _bf16(rng, *shape):
    bits = synth.bf16_round(rng.standard_normal(shape).astype(np.float32))
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t, synth.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("chunked", [True, False])
@pytest.mark.parametrize("B,s,H,Hkv,hd", [(512, 8192, 24, 8, 128), (512, 32768, 24, 8, 128),
                                          (1, 32768, 24, 8, 128), (130, 8000, 24, 8, 128),
                                          (700, 5000, 8, 2, 64)])
def test_long_prefix_attention_matches_oracle(B, s, H, Hkv, hd, chunked):
    """Long key ranges, spread over all SMs in equal chunks (with a
    workspace) or split over CTA pairs (without one)."""
    from dense_decoder_layer_gb300 import pds
    rng = np.random.default_rng(B + s)
    q, q64 = _bf16(rng, B, H, hd)
    k, k64 = _bf16(rng, s + B, Hkv, hd)
    v, v64 = _bf16(rng, s + B, Hkv, hd)
    o = torch.full((B, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = pds.pds_attention_workspace_bytes(B, s, H, hd) if chunked else 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    pds.pds_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, s, H, Hkv, hd,
                      stream, workspace=ws.data_ptr() if chunked else None,
                      workspace_bytes=ws_bytes)
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    want = oracle.causal_gqa_attention(q64, k64, v64, s).reshape(B, H * hd)
    assert_parity(bf16_to_f64(o), want, f"attention B={B} s={s} chunked={chunked}")


@pytest.mark.parametrize("s", [8192, 32768])
def test_long_prefix_stack_matches_oracle(s):
    """Two Llama-3.2-3B-shaped layers, 512 new rows over an s-row prefix."""
    dims = synth.Dims(2, 3072, 24, 8, 128, 8192, 512, s, 5.0e5)
    dims, (layers, pk, pv, hidden) = workload(dims)
    _check(run_gpu(dims, layers, pk, pv, hidden), oracle_result(dims), f"prefix {s}")
