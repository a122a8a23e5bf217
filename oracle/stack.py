"""Plain fp64 restatement of one prefill call through a run of dense layers.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (frink-models pages):

* ``src/fused_layer.rs`` (0.49.0), module doc "What it refuses": the
  layer is exactly ``x + ffn(rms_norm(x + branch))`` with a SwiGLU FFN of
  one dense expert, where ``branch`` is the attention of the
  pre-attention-normed ``x``.  The pre-FFN norm is a plain weighted RMS
  (``LayerFfnParts::for_layer``, the ``NormOp::Rms`` match).
* ``src/decoder/cuda_prefill.rs`` (0.29.0): module doc (a run of
  consecutive dense layers per call, seven matmuls per layer, each
  layer's K/V rows returned), ``try_cuda_prefill_dense_stack`` (SwiGLU
  only; one ``rms_eps`` for both norms; K/V rows pushed per layer, row
  ``b`` at ``b*kv_width``), ``cuda_prefill_layer`` (the descriptor's
  fields: two RMS gains, q/k/v/o/gate/up/down, the RoPE description,
  ``attn_scale = 1/sqrt(head_dim)``, the prefix as the cache's first
  ``start_pos`` rows, cache positions equal to ``start_pos``).
* ``src/decoder/device_attention.rs`` (0.38.0), doc of
  ``device_attention_layer``: q/k/v reach attention post-RoPE, the layer
  ends with ``wo``, the residual, the FFN norm, the FFN and the residual.

Readings where the pages are silent:
weights are ``[out, in]`` and ``y = x @ W.T``; RoPE is the NeoX-half
layout with ``omega_i = theta**(-2i/head_dim)`` over the full head;
query head ``h`` reads kv head ``h // (n_heads/n_kv_heads)``; new row
``b`` sits at position ``start_pos + b``; the K prefix is stored
post-RoPE and is not rotated again; RMSNorm is ``x/sqrt(mean(x^2)+eps)*g``.

Everything here is float64.  bf16 inputs are widened exactly.
"""

from __future__ import annotations

import numpy as np


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of an fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """Weighted RMSNorm over the last axis: ``x / sqrt(mean(x^2) + eps) * g``.

    fused_layer.rs, ``LayerFfnParts::for_layer``: the norm is "a plain
    weighted RMS"; cuda_prefill.rs, ``try_cuda_prefill_dense_stack``: one
    ``rms_eps`` serves both norms of the layer.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """``omega_i = theta**(-2i/head_dim)`` for ``i < head_dim/2`` (cuda_prefill.rs, ``LayerRopeCuda``: ``theta``, ``rot_dim`` = head_dim)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_neox(t: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate every head of ``t[n, heads, hd]`` by its row's position.

    NeoX layout (cuda_prefill.rs, ``RopeLayoutCuda::Neox``): channel ``i``
    pairs with channel ``i + hd/2``; the pair ``(u, w)`` turns by the angle
    ``p*omega_i`` into ``(u cos - w sin, u sin + w cos)``.
    """
    hd = t.shape[-1]
    half = hd // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    u, w = t[..., :half], t[..., half:]
    return np.concatenate([u * c - w * s, u * s + w * c], axis=-1)


def silu(t: np.ndarray) -> np.ndarray:
    """``t / (1 + exp(-t))`` (the SwiGLU gate; cuda_prefill.rs refuses every other activation)."""
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def causal_gqa_attention(q: np.ndarray, k_all: np.ndarray, v_all: np.ndarray,
                         start_pos: int) -> np.ndarray:
    """GQA causal attention of new rows over the cache prefix plus the new rows.

    ``q[B, H, hd]`` are the new rows at positions ``start_pos + b``;
    ``k_all``/``v_all`` are ``[start_pos + B, Hkv, hd]``: the prefix rows,
    then the new rows.  Row ``b`` sees keys ``j <= start_pos + b``; the
    scores are scaled by ``1/sqrt(hd)`` (cuda_prefill.rs, ``PrefillParams``:
    ``attn_scale``, no softcap, no window, ``prefix_k``/``prefix_v``).
    """
    B, H, hd = q.shape
    T, Hkv, _ = k_all.shape
    assert T == start_pos + B and H % Hkv == 0
    group = H // Hkv
    visible = np.arange(T)[None, :] <= (start_pos + np.arange(B))[:, None]   # [B, T]
    out = np.empty_like(q)
    for h in range(H):
        g = h // group
        z = (q[:, h, :] @ k_all[:, g, :].T) / np.sqrt(hd)
        z = np.where(visible, z, -np.inf)
        z = z - z.max(axis=1, keepdims=True)
        a = np.exp(z)
        a = a / a.sum(axis=1, keepdims=True)
        out[:, h, :] = a @ v_all[:, g, :]
    return out


def decoder_layer(x, w, k_prefix, v_prefix, start_pos, n_heads, n_kv_heads, head_dim,
                  rope_theta, rms_eps):
    """One dense layer: ``h = x + wo(attn(rms_norm(x)))``, ``x' = h + ffn(rms_norm(h))``.

    ``x`` is ``[B, d]`` float64.  ``w`` maps the tensor names of the layer
    to float64 arrays (matrices ``[out, in]``).  ``k_prefix``/``v_prefix``
    are float64 ``[start_pos, Hkv, hd]``.  Returns ``(x', k_rows, v_rows)``
    with the new rows ``[B, Hkv, hd]`` (K post-RoPE), the rows the call
    returns for each layer's cache (cuda_prefill.rs, the push loop of
    ``try_cuda_prefill_dense_stack``).
    """
    B = x.shape[0]
    pos = start_pos + np.arange(B)
    n = rms_norm(x, w["attn_norm"], rms_eps)
    q = (n @ w["wq"].T).reshape(B, n_heads, head_dim)
    k = (n @ w["wk"].T).reshape(B, n_kv_heads, head_dim)
    v = (n @ w["wv"].T).reshape(B, n_kv_heads, head_dim)
    q = rope_neox(q, pos, rope_theta)
    k = rope_neox(k, pos, rope_theta)
    k_all = np.concatenate([k_prefix, k], axis=0)
    v_all = np.concatenate([v_prefix, v], axis=0)
    o = causal_gqa_attention(q, k_all, v_all, start_pos).reshape(B, n_heads * head_dim)
    h = x + o @ w["wo"].T
    m = rms_norm(h, w["ffn_norm"], rms_eps)
    act = silu(m @ w["w_gate"].T) * (m @ w["w_up"].T)
    return h + act @ w["w_down"].T, k, v


def _widen_layer(raw: dict) -> dict:
    out = {}
    for name, t in raw.items():
        t = np.asarray(t)
        out[name] = widen_bf16(t) if t.dtype == np.uint16 else t.astype(np.float64)
    return out


def prefill_dense_stack(hidden, layers, prefix_k, prefix_v, start_pos, n_heads, n_kv_heads,
                        head_dim, rope_theta, rms_eps, n_layers=None):
    """A run of consecutive dense layers over one hidden batch.

    cuda_prefill.rs, module doc and ``try_cuda_prefill_dense_stack``: the
    batch passes through every layer of the run, and the call answers the
    new hidden batch plus each layer's new K/V rows.

    ``hidden`` float32/float64 ``[B, d]``; ``layers`` a list of per-layer
    dicts (bf16 bit matrices as uint16, float32 gains); ``prefix_k`` /
    ``prefix_v`` per-layer bf16 bits (or float) ``[start_pos, Hkv, hd]``.
    Weights are widened one layer at a time, so a large stack needs one
    layer of float64 at a time.  Returns ``(hidden_out, k_rows, v_rows)``,
    float64, with ``k_rows[l]``/``v_rows[l]`` of shape ``[B, Hkv, hd]``.
    """
    L = len(layers) if n_layers is None else n_layers
    x = np.asarray(hidden, dtype=np.float64)
    k_rows, v_rows = [], []
    for l in range(L):
        w = _widen_layer(layers[l])
        kp = prefix_k[l]
        vp = prefix_v[l]
        kp = widen_bf16(kp) if np.asarray(kp).dtype == np.uint16 else np.asarray(kp, np.float64)
        vp = widen_bf16(vp) if np.asarray(vp).dtype == np.uint16 else np.asarray(vp, np.float64)
        x, k, v = decoder_layer(x, w, kp, vp, start_pos, n_heads, n_kv_heads, head_dim,
                                rope_theta, rms_eps)
        k_rows.append(k)
        v_rows.append(v)
    return x, k_rows, v_rows
