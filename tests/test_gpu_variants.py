"""Parity of the optional parts of the launch (attention extras, RoPE
variants, softcap, sliding window) against the oracle, through the C ABI:
whole stacks, and the attention kernel alone."""

import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, bf16_to_f64, oracle_result, run_gpu, workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HD64 = synth.Dims(2, 512, 8, 2, 64, 1536, 130, 70, 1.0e4)
HD128 = synth.Dims(3, 768, 6, 2, 128, 2048, 200, 37, 5.0e5)

CASES = {
    # Qwen-style projections: q/k/v biases and per-head q/k norms
    "extras-hd128": (HD128, synth.Variant(extras=True)),
    "extras-hd64": (HD64, synth.Variant(extras=True)),
    # adjacent-pair layout, partial rotation
    "norm-layout-hd64": (HD64, synth.Variant(rope_layout="norm")),
    "norm-partial-hd128": (HD128, synth.Variant(rope_layout="norm", rot_dim=48)),
    # Neox over part of the head, frequency factors, scaled rotated channels
    "neox-partial-factors-mscale": (HD128, synth.Variant(rot_dim=64, freq_factors=True,
                                                         rope_mscale=1.25)),
    # the fast epilogue with frequency factors and a scale (table only)
    "factors-mscale-fast": (HD64, synth.Variant(freq_factors=True, rope_mscale=0.9)),
    # softcap and a window shorter than the key range
    "softcap-window": (HD128, synth.Variant(attn_softcap=2.0, window=100)),
    "window-hd64": (HD64, synth.Variant(window=64)),
    "everything": (HD64, synth.Variant(extras=True, rope_layout="norm", rot_dim=32,
                                       freq_factors=True, rope_mscale=1.1, attn_softcap=3.0,
                                       window=90)),
    # the general QKV epilogue on one row tile whose k range is split over a
    # cluster (row slices of 32: the last one ragged, or two of them empty)
    "extras-hd128-row-split": (HD128.replace(batch=100), synth.Variant(extras=True)),
    "everything-row-split": (HD64.replace(batch=60),
                             synth.Variant(extras=True, rope_layout="norm", rot_dim=32,
                                           freq_factors=True, rope_mscale=1.1,
                                           attn_softcap=3.0, window=90)),
}


def _check(got, want, tag):
    assert_parity(got[0], want[0], f"{tag} hidden_out")
    for l in range(len(want[1])):
        assert_parity(got[1][l], want[1][l], f"{tag} k_rows[{l}]")
        assert_parity(got[2][l], want[2][l], f"{tag} v_rows[{l}]")


@pytest.mark.parametrize("name", sorted(CASES))
def test_variant_stack_matches_oracle(name):
    dims, variant = CASES[name]
    dims, (layers, pk, pv, hidden) = workload(dims, 0, variant)
    want = oracle_result(dims, 0, None, variant)
    _check(run_gpu(dims, layers, pk, pv, hidden, variant=variant), want, name)


def test_full_size_variant_stack_matches_oracle():
    """The Llama-3.2-3B shape over its 1536-row prefix with every optional
    part on: biases, q/k norms, frequency factors, a 1024-position window
    (so whole key tiles are skipped and long ranges still split) and a
    softcap."""
    dims = synth.CONFIGS["llama3.2-3b-pp512-prefix1536"]
    variant = synth.Variant(extras=True, freq_factors=True, attn_softcap=30.0, window=1024)
    dims, (layers, pk, pv, hidden) = workload(dims, 0, variant)
    want = oracle_result(dims, 0, None, variant)
    _check(run_gpu(dims, layers, pk, pv, hidden, variant=variant), want, "3b-prefix-variant")


def _bf16(rng, *shape, scale=1.0):
    bits = synth.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t, synth.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("B,s,H,Hkv,hd,cap,win", [
    (130, 0, 8, 2, 64, 0.0, 1),        # window of one: every row its own value
    (130, 0, 8, 2, 64, 0.0, 100),
    (200, 333, 3, 1, 128, 0.0, 300),   # window reaching into the prefix
    (64, 100, 6, 2, 128, 2.0, 0),      # softcap alone (scores scaled up below)
    (512, 1536, 24, 8, 128, 30.0, 700),  # long ranges, split over CTA pairs
    (300, 1000, 4, 2, 64, 5.0, 1200),  # window longer than some rows' history
    (1, 77, 8, 8, 128, 1.5, 16),
    (512, 20000, 8, 2, 128, 20.0, 9000),  # long windowed ranges, chunked over all SMs
])
def test_attention_variants_match_oracle(B, s, H, Hkv, hd, cap, win):
    from dense_decoder_layer_gb300 import pds
    rng = np.random.default_rng(B + 13 * s + H + win)
    qs = 3.0 if cap else 1.0  # larger scores so that the cap bends them
    q, q64 = _bf16(rng, B, H, hd, scale=qs)
    k, k64 = _bf16(rng, s + B, Hkv, hd)
    v, v64 = _bf16(rng, s + B, Hkv, hd)
    o = torch.full((B, H * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = pds.pds_attention_workspace_bytes(B, s, H, hd)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    pds.pds_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, s, H, Hkv, hd,
                      stream, softcap=cap, window=win, workspace=ws.data_ptr(),
                      workspace_bytes=ws_bytes)
    assert pds.pds_component_sync(stream) == pds.PDS_OK
    want = oracle.causal_gqa_attention(q64, k64, v64, s, softcap=cap or None,
                                       window=win or None).reshape(B, H * hd)
    assert_parity(bf16_to_f64(o), want, f"attention B={B} s={s} cap={cap} window={win}")
