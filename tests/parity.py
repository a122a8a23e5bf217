"""Helpers of the GPU parity tests: tolerance checks and runs of both sides."""

from __future__ import annotations

import functools
import os

import numpy as np

import oracle
import synth

# Tolerance of every floating-point comparison against the oracle: relative
# L2 error <= 1e-2 and max-abs error <= 5e-2 * rms(oracle), on the hidden
# output and on every layer's K and V rows.
REL_L2 = 1e-2
MAX_ABS_RMS = 5e-2


def parity_stats(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    diff = got - want
    rms = float(np.sqrt(np.mean(want * want)))
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(want), 1e-300))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    return rel, mx, rms


def assert_parity(got, want, what="", rel_l2=REL_L2, max_abs_rms=MAX_ABS_RMS):
    rel, mx, rms = parity_stats(got, want)
    log = os.environ.get("PDS_PARITY_LOG")
    if log:  # one line per comparison: the margins behind the pass/fail
        with open(log, "a") as f:
            f.write(f"{what}\trel_l2 {rel:.4e}\tmax_abs/rms {mx / max(rms, 1e-300):.4e}\n")
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert rel <= rel_l2, f"{what}: relative L2 {rel:.3e} > {rel_l2}"
    assert mx <= max_abs_rms * rms, f"{what}: max-abs {mx:.3e} > {max_abs_rms}*rms ({rms:.3e})"
    return rel, mx, rms


def bf16_to_f64(t):
    """bf16 torch tensor (any device) -> float64 numpy."""
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def run_oracle(dims, layers, pk, pv, hidden, variant=synth.NO_VARIANT, seed=0):
    return oracle.prefill_dense_stack(hidden, layers, pk, pv, dims.start_pos, dims.n_heads,
                                      dims.n_kv_heads, dims.head_dim, dims.rope_theta,
                                      dims.rms_eps, **synth.variant_options(dims, variant, seed))


@functools.lru_cache(maxsize=4)
def workload(name_or_dims, seed=0, variant=synth.NO_VARIANT):
    dims = synth.CONFIGS[name_or_dims] if isinstance(name_or_dims, str) else name_or_dims
    return dims, synth.draw_workload(dims, seed, variant=variant)


@functools.lru_cache(maxsize=4)
def oracle_result(name_or_dims, seed=0, rows=None, variant=synth.NO_VARIANT):
    """Oracle on the workload, optionally on its first `rows` rows only
    (exact for those rows: row b depends on rows <= b only)."""
    dims, (layers, pk, pv, hidden) = workload(name_or_dims, seed, variant)
    if rows is not None:
        dims = dims.replace(batch=rows)
        hidden = hidden[:rows]
    return run_oracle(dims, layers, pk, pv, hidden, variant, seed)


def run_gpu(dims, layers, pk, pv, hidden, extra_capacity=0, variant=synth.NO_VARIANT, seed=0):
    """One host-I/O call of the CUDA stack; returns (hidden_out, [k], [v]) as float64."""
    import torch
    from dense_decoder_layer_gb300.stack import DenseStack
    st = DenseStack(dims, dims.start_pos + dims.batch + extra_capacity, dims.batch,
                    variant=variant, freq_factors=synth.draw_freq_factors(dims, variant, seed))
    st.load_layers(layers)
    st.load_prefix(pk, pv)
    out = st.prefill(torch.from_numpy(np.ascontiguousarray(hidden, np.float32)), dims.start_pos)
    ks, vs = [], []
    for l in range(dims.n_layers):
        k, v = st.rows(l, dims.start_pos, dims.batch)
        ks.append(bf16_to_f64(k))
        vs.append(bf16_to_f64(v))
    res = (out.numpy().astype(np.float64), ks, vs)
    st.close()
    return res
