"""PyTorch-side owner of the buffers of one prefill stack.

PyTorch provides device memory and streams; every step of the call runs
in ``libpds.so`` through :mod:`.pds`.  ``DenseStack`` keeps the weight
tensors, the per-layer K/V caches and the workspace alive and hands their
pointers to the C ABI.
"""

from __future__ import annotations

import numpy as np
import torch

from . import pds

LAYER_FIELDS = pds.LAYER_FIELDS
EXTRA_FIELDS = pds.EXTRA_FIELDS
# pds_layer field -> tensor name of a drawn layer (synth.LAYER_TENSORS)
SYNTH_NAMES = {"attn_norm_w": "attn_norm", "ffn_norm_w": "ffn_norm"}


def _bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """bf16 bit patterns (uint16 numpy) -> bf16 torch tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device, non_blocking=False)


class DenseStack:
    """A run of ``n_layers`` dense layers on one GPU, with its caches.

    ``dims`` is any object with the model fields of ``pds_dims`` (n_layers,
    d_model, n_heads, n_kv_heads, head_dim, ffn_dim, rope_theta, rms_eps);
    ``variant`` optionally gives the run-wide RoPE / attention options
    (rope_layout, rot_dim, rope_mscale, attn_softcap, window) and
    ``freq_factors`` the RoPE frequency factors.
    """

    def __init__(self, dims, cache_capacity: int, max_batch: int, device="cuda", variant=None,
                 freq_factors=None):
        self.dims = dims
        self.device = torch.device(device)
        self.cache_capacity = int(cache_capacity)
        self.max_batch = int(max_batch)
        self.plan = pds.pds_plan_create(pds.make_dims(dims, variant, freq_factors))
        kvw = dims.n_kv_heads * dims.head_dim
        L = dims.n_layers
        self.k_cache = [torch.zeros(self.cache_capacity, kvw, dtype=torch.bfloat16,
                                    device=self.device) for _ in range(L)]
        self.v_cache = [torch.zeros_like(self.k_cache[0]) for _ in range(L)]
        # the C arrays of pointers are built once, not on every call
        self._k_ptrs = pds._ptrs([t.data_ptr() for t in self.k_cache])
        self._v_ptrs = pds._ptrs([t.data_ptr() for t in self.v_cache])
        # room for the attention's chunked key ranges up to the cache's capacity
        self.ws_bytes = pds.pds_workspace_bytes(self.plan, self.max_batch,
                                                max(0, self.cache_capacity - 1))
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.weights = []
        self._layer_ptrs = []
        self._layers_c = pds._layer_array([])

    def close(self):
        if self.plan is not None:
            pds.pds_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ weights
    def load_layers(self, layers) -> None:
        """``layers``: per-layer dicts of numpy arrays (bf16 bits uint16 for
        matrices, float32 for the gains and the optional extras), as
        :func:`synth.draw_workload` makes."""
        self.weights, self._layer_ptrs = [], []
        for l in layers:
            t = {}
            for n in LAYER_FIELDS + EXTRA_FIELDS:
                a = l.get(n, l.get(SYNTH_NAMES.get(n, ""), None))
                if a is None:
                    continue
                if a.dtype == np.uint16:
                    t[n] = _bf16_tensor(a, self.device)
                else:
                    t[n] = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(self.device)
            self.weights.append(t)
            self._layer_ptrs.append({n: t[n].data_ptr() for n in t})
        self._layers_c = pds._layer_array(self._layer_ptrs)

    def set_layer_tensors(self, layers) -> None:
        """Use device tensors the caller already holds (dicts field -> tensor)."""
        self.weights = list(layers)
        self._layer_ptrs = [{n: l[n].data_ptr() for n in LAYER_FIELDS + EXTRA_FIELDS if n in l}
                            for l in layers]
        self._layers_c = pds._layer_array(self._layer_ptrs)

    def load_prefix(self, prefix_k, prefix_v) -> None:
        """Rows [0, s) of every cache from bf16 bit arrays [s, Hkv, hd]."""
        for l in range(self.dims.n_layers):
            s = prefix_k[l].shape[0]
            if s:
                self.k_cache[l][:s].copy_(_bf16_tensor(prefix_k[l].reshape(s, -1), self.device))
                self.v_cache[l][:s].copy_(_bf16_tensor(prefix_v[l].reshape(s, -1), self.device))

    # --------------------------------------------------------------- calls
    def _stream(self, stream):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return s.cuda_stream

    def prefill(self, hidden: torch.Tensor, start_pos: int, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
        """Host float32 [B, d] in, host float32 [B, d] out (blocking)."""
        assert hidden.device.type == "cpu" and hidden.dtype == torch.float32
        hidden = hidden.contiguous()
        B = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        pds.pds_prefill_dense_stack(
            self.plan, self._layers_c, self._k_ptrs, self._v_ptrs, self.cache_capacity,
            start_pos, B,
            hidden.data_ptr(), out.data_ptr(), self.workspace.data_ptr(), self.ws_bytes,
            self._stream(stream))
        return out

    def prefill_device(self, hidden: torch.Tensor, start_pos: int, out: torch.Tensor,
                       stream=None) -> None:
        """Device float32 [B, d] in and out, enqueued on the stream."""
        B = hidden.shape[0]
        pds.pds_prefill_dense_stack_device(
            self.plan, self._layers_c, self._k_ptrs, self._v_ptrs, self.cache_capacity,
            start_pos, B,
            hidden.data_ptr(), out.data_ptr(), self.workspace.data_ptr(), self.ws_bytes,
            self._stream(stream))

    def sync(self, stream=None) -> None:
        pds.pds_plan_sync(self.plan, self._stream(stream))

    def rows(self, l: int, start_pos: int, batch: int):
        """Layer l's new K and V rows of the last call, bf16 [B, Hkv, hd] views."""
        shp = (batch, self.dims.n_kv_heads, self.dims.head_dim)
        return (self.k_cache[l][start_pos:start_pos + batch].view(shp),
                self.v_cache[l][start_pos:start_pos + batch].view(shp))
