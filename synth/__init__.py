"""Seeded synthetic inputs for the dense decoder-layer prefill stack.

This module is shared by the CPU oracle and by the CUDA path's tests and
benchmark.  It holds none of the layer arithmetic: it only draws the
random tensors of a workload and rounds the ones that are stored as bf16.

Recipe (the workloads of the dense prefill stack; the pages give the
shapes and the distributions, the generator choice is ours):

* matrices ``W[out, in]`` ~ N(0, 1/in), drawn in float32, then rounded to
  bf16 (round-to-nearest-even); ``in`` is ``d`` for wq/wk/wv/gate/up,
  ``n_heads*head_dim`` for wo and ``ffn`` for down;
* RMSNorm gains ``1 + 0.1*N(0,1)`` in float32 (kept in float32);
* hidden batch ``[B, d]`` ~ N(0,1) in float32;
* K/V prefix per layer ``[start_pos, n_kv_heads, head_dim]`` ~ N(0,1)
  rounded to bf16.  The K prefix is taken as already rotated (a rotation
  of an isotropic Gaussian pair is again an isotropic Gaussian pair, so
  drawing the rotated values directly gives the same distribution).
* optional attention extras per layer (float32): q/k/v biases ~ N(0, 0.5^2),
  q/k norm gains ``1 + 0.1*N(0,1)`` of ``[head_dim]``;
* optional RoPE frequency factors ``1 + 3*U[0,1)`` per rotated pair
  (float32), drawn once per workload.

Every tensor has its own PCG64 stream, keyed by ``(seed, layer, tensor
id)``, so tensors can be drawn in parallel threads and a subset of the
layers (or a prefix of the rows of the hidden batch) can be drawn without
drawing the rest.  The hidden batch is drawn row-major from its own
stream, so its first ``b`` rows do not depend on the total batch size.
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

__all__ = [
    "Dims",
    "Variant",
    "NO_VARIANT",
    "EXTRA_TENSORS",
    "draw_extras",
    "draw_freq_factors",
    "variant_options",
    "CONFIGS",
    "LAYER_TENSORS",
    "bf16_round",
    "bf16_bits_to_f32",
    "draw_layer",
    "draw_hidden",
    "draw_prefix",
    "draw_workload",
]


@dataclasses.dataclass(frozen=True)
class Dims:
    """Shape of a dense Llama-style stack and of one prefill call."""

    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    batch: int          # B, new tokens of the call
    start_pos: int      # s, rows already in each layer's K/V cache
    rope_theta: float
    rms_eps: float = 1e-5

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "Dims":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Variant:
    """The optional parts of a run: attention extras (per layer) and the
    RoPE / attention options (the same for every layer of the run)."""

    extras: bool = False          # q/k/v biases and q/k norm gains in every layer
    rope_layout: str = "neox"     # "neox" or "norm"
    rot_dim: int = 0              # 0: the whole head
    freq_factors: bool = False    # draw frequency factors
    rope_mscale: float = 1.0
    attn_softcap: float = 0.0     # 0: none
    window: int = 0               # 0: none


NO_VARIANT = Variant()


# The workloads of the dense prefill stack, by what they are.
CONFIGS = {
    "tiny": Dims(2, 256, 4, 2, 64, 768, 8, 0, 1.0e4),
    "llama3.2-1b": Dims(16, 2048, 32, 8, 64, 8192, 128, 0, 5.0e5),
    "llama3.2-3b-pp512": Dims(28, 3072, 24, 8, 128, 8192, 512, 0, 5.0e5),
    "llama3.2-3b-pp512-prefix1536": Dims(28, 3072, 24, 8, 128, 8192, 512, 1536, 5.0e5),
    "llama3-8b-pp2048-prefix2048": Dims(32, 4096, 32, 8, 128, 14336, 2048, 2048, 5.0e5),
    # decode steps against a resident 2048-row cache (the matvec regime)
    "llama3.2-3b-decode-b1-ctx2048": Dims(28, 3072, 24, 8, 128, 8192, 1, 2048, 5.0e5),
    "llama3.2-3b-decode-b8-ctx2048": Dims(28, 3072, 24, 8, 128, 8192, 8, 2048, 5.0e5),
    # long cached prefixes (attention-dominated prefill)
    "llama3.2-3b-pp512-prefix8192": Dims(28, 3072, 24, 8, 128, 8192, 512, 8192, 5.0e5),
    "llama3.2-3b-pp512-prefix32768": Dims(28, 3072, 24, 8, 128, 8192, 512, 32768, 5.0e5),
}

# Tensor ids of one layer, in a fixed order (the id keys the stream).
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
_PREFIX_K, _PREFIX_V = 9, 10
EXTRA_TENSORS = ("q_bias", "k_bias", "v_bias", "q_norm", "k_norm")
_EXTRA_IDS = {n: 11 + i for i, n in enumerate(EXTRA_TENSORS)}
_FREQ_FACTORS = 16
_HIDDEN_LAYER = 0xFFFF


def _rng(seed: int, layer: int, tid: int) -> np.random.Generator:
    return np.random.default_rng([seed, layer, tid])


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even.

    Inputs are finite (Gaussian draws), so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _shape_of(dims: Dims, name: str):
    d, qw, kvw, f = dims.d_model, dims.q_width, dims.kv_width, dims.ffn_dim
    return {
        "attn_norm": (d,),
        "ffn_norm": (d,),
        "wq": (qw, d),
        "wk": (kvw, d),
        "wv": (kvw, d),
        "wo": (d, qw),
        "w_gate": (f, d),
        "w_up": (f, d),
        "w_down": (d, f),
    }[name]


def _draw_tensor(seed: int, layer: int, dims: Dims, name: str) -> np.ndarray:
    tid = LAYER_TENSORS.index(name)
    shape = _shape_of(dims, name)
    g = _rng(seed, layer, tid)
    if name.endswith("_norm"):
        z = g.standard_normal(shape, dtype=np.float32)
        return (np.float32(1.0) + np.float32(0.1) * z).astype(np.float32)
    z = np.empty(shape, dtype=np.float32)
    g.standard_normal(out=z, dtype=np.float32)
    z *= np.float32(1.0 / np.sqrt(shape[1]))
    return bf16_round(z)


def _pool(threads):
    n = threads or min(32, os.cpu_count() or 1)
    return _cf.ThreadPoolExecutor(max_workers=n)


def draw_layer(dims: Dims, layer: int, seed: int = 0, threads: int | None = None) -> dict:
    """One layer's tensors: norms float32 ``[d]``, matrices bf16 bits ``[out, in]``."""
    with _pool(threads) as ex:
        futs = {n: ex.submit(_draw_tensor, seed, layer, dims, n) for n in LAYER_TENSORS}
        return {n: f.result() for n, f in futs.items()}


def draw_hidden(dims: Dims, seed: int = 0, rows: int | None = None) -> np.ndarray:
    """Hidden batch ``[rows or B, d]`` float32; row b is the same for every B."""
    rows = dims.batch if rows is None else rows
    g = _rng(seed, _HIDDEN_LAYER, 0)
    return g.standard_normal((rows, dims.d_model), dtype=np.float32)


def draw_prefix(dims: Dims, layer: int, seed: int = 0):
    """K and V prefix of one layer, bf16 bits ``[start_pos, n_kv_heads, head_dim]``."""
    shape = (dims.start_pos, dims.n_kv_heads, dims.head_dim)
    out = []
    for tid in (_PREFIX_K, _PREFIX_V):
        g = _rng(seed, layer, tid)
        out.append(bf16_round(g.standard_normal(shape, dtype=np.float32)))
    return out[0], out[1]


def draw_extras(dims: Dims, layer: int, seed: int = 0) -> dict:
    """One layer's attention extras (float32): biases ``[H*hd]``/``[Hkv*hd]``
    ~ N(0, 0.5^2) and q/k norm gains ``[hd]`` = 1 + 0.1*N(0,1)."""
    shapes = {"q_bias": dims.q_width, "k_bias": dims.kv_width, "v_bias": dims.kv_width,
              "q_norm": dims.head_dim, "k_norm": dims.head_dim}
    out = {}
    for n in EXTRA_TENSORS:
        z = _rng(seed, layer, _EXTRA_IDS[n]).standard_normal(shapes[n], dtype=np.float32)
        if n.endswith("_norm"):
            out[n] = (np.float32(1.0) + np.float32(0.1) * z).astype(np.float32)
        else:
            out[n] = (np.float32(0.5) * z).astype(np.float32)
    return out


def draw_freq_factors(dims: Dims, variant: Variant, seed: int = 0):
    """RoPE frequency factors ``1 + 3*U[0,1)`` per rotated pair (float32), or None."""
    if not variant.freq_factors:
        return None
    pairs = (variant.rot_dim or dims.head_dim) // 2
    u = _rng(seed, _HIDDEN_LAYER, _FREQ_FACTORS).random(pairs, dtype=np.float32)
    return (np.float32(1.0) + np.float32(3.0) * u).astype(np.float32)


def variant_options(dims: Dims, variant: Variant, seed: int = 0) -> dict:
    """The run-wide options of a variant as keyword arguments (oracle names)."""
    return dict(rope_layout=variant.rope_layout, rot_dim=variant.rot_dim or None,
                freq_factors=draw_freq_factors(dims, variant, seed),
                rope_mscale=variant.rope_mscale, attn_softcap=variant.attn_softcap or None,
                window=variant.window or None)


def draw_workload(dims: Dims, seed: int = 0, threads: int | None = None,
                  variant: Variant = NO_VARIANT):
    """All inputs of one call.

    Returns ``(layers, prefix_k, prefix_v, hidden)`` with ``layers`` a list
    of per-layer dicts (see :func:`draw_layer`), ``prefix_k``/``prefix_v``
    lists of per-layer bf16 bit arrays and ``hidden`` float32 ``[B, d]``.
    """
    with _pool(threads) as ex:
        futs = [[ex.submit(_draw_tensor, seed, l, dims, n) for n in LAYER_TENSORS]
                for l in range(dims.n_layers)]
        pfx = [ex.submit(draw_prefix, dims, l, seed) for l in range(dims.n_layers)]
        layers = [{n: f.result() for n, f in zip(LAYER_TENSORS, fl)} for fl in futs]
        pk = [p.result()[0] for p in pfx]
        pv = [p.result()[1] for p in pfx]
    if variant.extras:
        for l, w in enumerate(layers):
            w.update(draw_extras(dims, l, seed))
    return layers, pk, pv, draw_hidden(dims, seed)
