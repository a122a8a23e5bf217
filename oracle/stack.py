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

The launch descriptor of cuda_prefill.rs also carries optional parts, all
off by default here and read as follows (the pages name them, they do not
print their arithmetic):

* ``AttnExtrasCuda``: ``q_bias``/``k_bias``/``v_bias`` are added to the
  projections; ``q_norm``/``k_norm`` are per-head RMSNorm gains ``[hd]``
  applied to every head of q and k (with the layer's ``rms_eps``) after the
  bias and before RoPE.
* ``LayerRopeCuda``: ``layout`` Neox pairs channel ``i`` with
  ``i + rot_dim/2``, Norm pairs ``2i`` with ``2i+1``; only the first
  ``rot_dim`` channels of a head turn; ``freq_factors[i]`` divides the
  angular frequency of pair ``i``; ``mscale`` multiplies the rotated
  channels (cos and sin).
* ``PrefillParams``: ``attn_softcap`` caps the scaled score ``z`` as
  ``cap*tanh(z/cap)``; ``window`` lets the row at position ``p`` see keys
  ``j`` with ``p - window < j <= p`` only.

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


def rope_inv_freq(rot_dim: int, theta: float, freq_factors=None) -> np.ndarray:
    """``omega_i = theta**(-2i/rot_dim) / freq_factors[i]`` for ``i < rot_dim/2``.

    cuda_prefill.rs, ``LayerRopeCuda``: ``theta``, ``rot_dim`` (the head
    width when absent) and ``freq_factors`` (none: every factor is 1).
    """
    i = np.arange(rot_dim // 2, dtype=np.float64)
    omega = np.power(float(theta), -2.0 * i / rot_dim)
    if freq_factors is not None:
        omega = omega / np.asarray(freq_factors, dtype=np.float64)
    return omega


def rope_neox(t: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate every head of ``t[n, heads, hd]`` by its row's position.

    NeoX layout (cuda_prefill.rs, ``RopeLayoutCuda::Neox``): channel ``i``
    pairs with channel ``i + hd/2``; the pair ``(u, w)`` turns by the angle
    ``p*omega_i`` into ``(u cos - w sin, u sin + w cos)``.
    """
    return rope_rotate(t, positions, theta)


def rope_rotate(t: np.ndarray, positions: np.ndarray, theta: float, layout: str = "neox",
                rot_dim: int | None = None, freq_factors=None, mscale: float = 1.0) -> np.ndarray:
    """RoPE of every head of ``t[n, heads, hd]`` at its row's position.

    cuda_prefill.rs, ``LayerRopeCuda`` / ``RopeLayoutCuda``: the first
    ``rot_dim`` channels of a head form ``rot_dim/2`` pairs, pair ``i``
    being channels ``(i, i + rot_dim/2)`` in the Neox layout and
    ``(2i, 2i+1)`` in the Norm layout; pair ``(u, w)`` turns by ``p*omega_i``
    into ``mscale*(u cos - w sin, u sin + w cos)``; channels from ``rot_dim``
    on are left as they are.
    """
    hd = t.shape[-1]
    rot = hd if rot_dim is None else int(rot_dim)
    half = rot // 2
    ang = (np.asarray(positions, dtype=np.float64)[:, None]
           * rope_inv_freq(rot, theta, freq_factors)[None, :])
    c = mscale * np.cos(ang)[:, None, :]
    s = mscale * np.sin(ang)[:, None, :]
    out = np.array(t, dtype=np.float64, copy=True)
    if layout == "neox":
        u, w = t[..., :half], t[..., half:rot]
        out[..., :half] = u * c - w * s
        out[..., half:rot] = u * s + w * c
    elif layout == "norm":
        u, w = t[..., 0:rot:2], t[..., 1:rot:2]
        out[..., 0:rot:2] = u * c - w * s
        out[..., 1:rot:2] = u * s + w * c
    else:
        raise ValueError(f"unknown RoPE layout {layout!r}")
    return out


def silu(t: np.ndarray) -> np.ndarray:
    """``t / (1 + exp(-t))`` (the SwiGLU gate; cuda_prefill.rs refuses every other activation)."""
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def causal_gqa_attention(q: np.ndarray, k_all: np.ndarray, v_all: np.ndarray,
                         start_pos: int, softcap: float | None = None,
                         window: int | None = None) -> np.ndarray:
    """GQA causal attention of new rows over the cache prefix plus the new rows.

    ``q[B, H, hd]`` are the new rows at positions ``start_pos + b``;
    ``k_all``/``v_all`` are ``[start_pos + B, Hkv, hd]``: the prefix rows,
    then the new rows.  Row ``b`` sees keys ``j <= start_pos + b``; the
    scores are scaled by ``1/sqrt(hd)`` (cuda_prefill.rs, ``PrefillParams``:
    ``attn_scale``, ``prefix_k``/``prefix_v``).  ``softcap`` (``attn_softcap``)
    replaces a scaled score ``z`` by ``softcap*tanh(z/softcap)``; ``window``
    hides the keys ``j <= p - window`` from the row at position ``p``.
    """
    B, H, hd = q.shape
    T, Hkv, _ = k_all.shape
    assert T == start_pos + B and H % Hkv == 0
    group = H // Hkv
    pos = start_pos + np.arange(B)
    visible = np.arange(T)[None, :] <= pos[:, None]   # [B, T]
    if window is not None:
        visible &= np.arange(T)[None, :] > (pos - window)[:, None]
    out = np.empty_like(q)
    for h in range(H):
        g = h // group
        z = (q[:, h, :] @ k_all[:, g, :].T) / np.sqrt(hd)
        if softcap is not None:
            z = softcap * np.tanh(z / softcap)
        z = np.where(visible, z, -np.inf)
        z = z - z.max(axis=1, keepdims=True)
        a = np.exp(z)
        a = a / a.sum(axis=1, keepdims=True)
        out[:, h, :] = a @ v_all[:, g, :]
    return out


def decoder_layer(x, w, k_prefix, v_prefix, start_pos, n_heads, n_kv_heads, head_dim,
                  rope_theta, rms_eps, rope_layout="neox", rot_dim=None, freq_factors=None,
                  rope_mscale=1.0, attn_softcap=None, window=None):
    """One dense layer: ``h = x + wo(attn(rms_norm(x)))``, ``x' = h + ffn(rms_norm(h))``.

    ``x`` is ``[B, d]`` float64.  ``w`` maps the tensor names of the layer
    to float64 arrays (matrices ``[out, in]``); the optional attention
    extras ``q_bias``, ``k_bias``, ``v_bias`` (``[H*hd]``, ``[Hkv*hd]``) and
    ``q_norm``, ``k_norm`` (``[hd]``) are used when present
    (cuda_prefill.rs, ``AttnExtrasCuda``).  ``k_prefix``/``v_prefix`` are
    float64 ``[start_pos, Hkv, hd]``.  Returns ``(x', k_rows, v_rows)`` with
    the new rows ``[B, Hkv, hd]`` (K post-RoPE), the rows the call returns
    for each layer's cache (cuda_prefill.rs, the push loop of
    ``try_cuda_prefill_dense_stack``).
    """
    B = x.shape[0]
    pos = start_pos + np.arange(B)
    n = rms_norm(x, w["attn_norm"], rms_eps)
    q = n @ w["wq"].T
    k = n @ w["wk"].T
    v = n @ w["wv"].T
    if w.get("q_bias") is not None:
        q = q + w["q_bias"]
    if w.get("k_bias") is not None:
        k = k + w["k_bias"]
    if w.get("v_bias") is not None:
        v = v + w["v_bias"]
    q = q.reshape(B, n_heads, head_dim)
    k = k.reshape(B, n_kv_heads, head_dim)
    v = v.reshape(B, n_kv_heads, head_dim)
    if w.get("q_norm") is not None:
        q = rms_norm(q, w["q_norm"], rms_eps)
    if w.get("k_norm") is not None:
        k = rms_norm(k, w["k_norm"], rms_eps)
    rope = dict(layout=rope_layout, rot_dim=rot_dim, freq_factors=freq_factors,
                mscale=rope_mscale)
    q = rope_rotate(q, pos, rope_theta, **rope)
    k = rope_rotate(k, pos, rope_theta, **rope)
    k_all = np.concatenate([k_prefix, k], axis=0)
    v_all = np.concatenate([v_prefix, v], axis=0)
    o = causal_gqa_attention(q, k_all, v_all, start_pos, softcap=attn_softcap,
                             window=window).reshape(B, n_heads * head_dim)
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
                        head_dim, rope_theta, rms_eps, n_layers=None, **variants):
    """A run of consecutive dense layers over one hidden batch.

    cuda_prefill.rs, module doc and ``try_cuda_prefill_dense_stack``: the
    batch passes through every layer of the run, and the call answers the
    new hidden batch plus each layer's new K/V rows.

    ``hidden`` float32/float64 ``[B, d]``; ``layers`` a list of per-layer
    dicts (bf16 bit matrices as uint16, float32 gains); ``prefix_k`` /
    ``prefix_v`` per-layer bf16 bits (or float) ``[start_pos, Hkv, hd]``.
    Weights are widened one layer at a time, so a large stack needs one
    layer of float64 at a time.  ``variants`` are the keyword options of
    :func:`decoder_layer` (RoPE layout and its parts, softcap, window), the
    same for every layer of the run.  Returns ``(hidden_out, k_rows,
    v_rows)``, float64, with ``k_rows[l]``/``v_rows[l]`` of shape
    ``[B, Hkv, hd]``.
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
                                rope_theta, rms_eps, **variants)
        k_rows.append(k)
        v_rows.append(v)
    return x, k_rows, v_rows
