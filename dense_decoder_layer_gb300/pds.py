"""ctypes binding of ``libpds.so`` (the C ABI in ``include/pds.h``).

Argument marshalling only: every step of the prefill stack runs in the
library's CUDA kernels.  The functions keep the C names; tensors are
passed as device pointers (``tensor.data_ptr()``) and streams as
``torch.cuda.Stream.cuda_stream`` handles.  A missing library is an
error: there is no other implementation of these calls.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpds.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pds.h")

PDS_OK, PDS_DECLINED, PDS_EINVAL, PDS_ELAUNCH, PDS_ETIMEOUT, PDS_ENOMEM = range(6)
STATUS_NAMES = {0: "PDS_OK", 1: "PDS_DECLINED", 2: "PDS_EINVAL", 3: "PDS_ELAUNCH",
                4: "PDS_ETIMEOUT", 5: "PDS_ENOMEM"}


class PdsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


PDS_ROPE_NEOX, PDS_ROPE_NORM = 0, 1


class pds_dims(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("rope_layout", ctypes.c_int32), ("rot_dim", ctypes.c_int32),
                ("freq_factors", ctypes.POINTER(ctypes.c_float)),
                ("rope_mscale", ctypes.c_float), ("attn_softcap", ctypes.c_float),
                ("window", ctypes.c_int32)]


LAYER_FIELDS = ("attn_norm_w", "ffn_norm_w", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")
EXTRA_FIELDS = ("q_bias", "k_bias", "v_bias", "q_norm", "k_norm")


class pds_layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS + EXTRA_FIELDS]


KERNEL_KINDS = ("prep", "qkv", "attn", "wo", "gateup", "down")


class pds_kernel_times(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * len(KERNEL_KINDS)),
                ("total_ms", ctypes.c_double * len(KERNEL_KINDS))]


_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree library (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first")
    try:  # share torch's CUDA runtime when torch is present
        import torch  # noqa: F401
    except ImportError:
        pass
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "pds_plan_create": (st, [ctypes.POINTER(pds_dims), ctypes.POINTER(ctypes.c_void_p)]),
        "pds_plan_destroy": (None, [vp]),
        "pds_workspace_bytes": (sz, [vp, i32, i32]),
        "pds_prefill_dense_stack": (st, [vp, ctypes.POINTER(pds_layer), pp, pp, i32, i32, i32,
                                         vp, vp, vp, sz, vp]),
        "pds_prefill_dense_stack_device": (st, [vp, ctypes.POINTER(pds_layer), pp, pp, i32, i32,
                                                i32, vp, vp, vp, sz, vp]),
        "pds_plan_sync": (st, [vp, vp]),
        "pds_last_error": (ctypes.c_char_p, []),
        "pds_gemm_bf16": (st, [vp, vp, vp, i32, i32, i32, vp, sz, vp]),
        "pds_gemm_workspace_bytes": (sz, [i32, i32]),
        "pds_gemm_bf16_noalloc": (st, [vp, vp, vp, i32, i32, i32, vp]),
        "pds_attention": (st, [vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                               vp, sz, vp]),
        "pds_attention_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "pds_plan_set_timing": (st, [vp, i32]),
        "pds_selftest_stuck_wait": (st, [ctypes.c_uint32, vp]),
        "pds_component_sync": (st, [vp]),
        "pds_plan_kernel_times": (st, [vp, vp, ctypes.POINTER(pds_kernel_times), i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def header_functions() -> list[str]:
    """Names of the functions ``include/pds.h`` declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pds_[a-z0-9_]+)\s*\(", text)))


def last_error() -> str:
    return load().pds_last_error().decode()


def check(status: int) -> None:
    if status != PDS_OK:
        raise PdsError(status, last_error())


def _ptrs(values):
    if isinstance(values, ctypes.Array):  # already marshalled (see DenseStack)
        return values
    arr = (ctypes.c_void_p * len(values))()
    for i, v in enumerate(values):
        arr[i] = v
    return arr


# -------------------------------------------------------- C-named wrappers

def pds_plan_create(dims: pds_dims) -> ctypes.c_void_p:
    plan = ctypes.c_void_p()
    check(load().pds_plan_create(ctypes.byref(dims), ctypes.byref(plan)))
    return plan


def pds_plan_destroy(plan) -> None:
    load().pds_plan_destroy(plan)


def pds_workspace_bytes(plan, max_batch: int, max_start_pos: int = 0) -> int:
    return load().pds_workspace_bytes(plan, max_batch, max_start_pos)


def _layer_array(layers):
    if isinstance(layers, ctypes.Array):  # already marshalled (see DenseStack)
        return layers
    arr = (pds_layer * len(layers))()
    for i, l in enumerate(layers):
        for n in LAYER_FIELDS + EXTRA_FIELDS:
            setattr(arr[i], n, l.get(n))
    return arr


def pds_prefill_dense_stack(plan, layers, k_cache, v_cache, cache_capacity, start_pos, batch,
                            hidden_in, hidden_out, workspace, workspace_bytes, stream) -> None:
    """Host in/out call.  ``layers``: list of dicts field -> device pointer;
    ``k_cache``/``v_cache``: lists of device pointers (or the ctypes arrays that
    ``_layer_array`` / ``_ptrs`` make); ``hidden_in``/``hidden_out``:
    host pointers."""
    check(load().pds_prefill_dense_stack(plan, _layer_array(layers), _ptrs(k_cache),
                                         _ptrs(v_cache), cache_capacity, start_pos, batch,
                                         hidden_in, hidden_out, workspace, workspace_bytes,
                                         stream))


def pds_prefill_dense_stack_device(plan, layers, k_cache, v_cache, cache_capacity, start_pos,
                                   batch, hidden_in_dev, hidden_out_dev, workspace,
                                   workspace_bytes, stream) -> None:
    check(load().pds_prefill_dense_stack_device(plan, _layer_array(layers), _ptrs(k_cache),
                                                _ptrs(v_cache), cache_capacity, start_pos, batch,
                                                hidden_in_dev, hidden_out_dev, workspace,
                                                workspace_bytes, stream))


def pds_plan_sync(plan, stream) -> None:
    check(load().pds_plan_sync(plan, stream))


def pds_gemm_workspace_bytes(M: int, N: int) -> int:
    return load().pds_gemm_workspace_bytes(M, N)


def pds_gemm_bf16(A, W, C, M, N, K, workspace, workspace_bytes, stream) -> None:
    check(load().pds_gemm_bf16(A, W, C, M, N, K, workspace, workspace_bytes, stream))


def pds_gemm_bf16_noalloc(A, W, C, M, N, K, stream) -> None:
    check(load().pds_gemm_bf16_noalloc(A, W, C, M, N, K, stream))


def pds_attention(q, k, v, o, batch, start_pos, n_heads, n_kv_heads, head_dim, stream,
                  softcap: float = 0.0, window: int = 0, workspace=None,
                  workspace_bytes: int = 0) -> None:
    check(load().pds_attention(q, k, v, o, batch, start_pos, n_heads, n_kv_heads, head_dim,
                               softcap, window, workspace, workspace_bytes if workspace else 0,
                               stream))


def pds_attention_workspace_bytes(batch, start_pos, n_heads, head_dim) -> int:
    return load().pds_attention_workspace_bytes(batch, start_pos, n_heads, head_dim)


def pds_plan_set_timing(plan, enable: bool) -> None:
    check(load().pds_plan_set_timing(plan, 1 if enable else 0))


def pds_plan_kernel_times(plan, stream, reset: bool = False) -> dict:
    """{kind: (launches, total_ms)} accumulated since the last reset."""
    kt = pds_kernel_times()
    check(load().pds_plan_kernel_times(plan, stream, ctypes.byref(kt), 1 if reset else 0))
    return {k: (kt.launches[i], kt.total_ms[i]) for i, k in enumerate(KERNEL_KINDS)}


def pds_selftest_stuck_wait(limit_us: int, stream) -> None:
    """Enqueue the bounded-wait self test (its timeout shows in pds_component_sync)."""
    check(load().pds_selftest_stuck_wait(limit_us, stream))


def pds_component_sync(stream) -> int:
    """Status of the component calls since the last sync (PDS_OK or PDS_ETIMEOUT);
    other failures raise."""
    st = load().pds_component_sync(stream)
    if st not in (PDS_OK, PDS_ETIMEOUT):
        raise PdsError(st, last_error())
    return st


def make_dims(dims, variant=None, freq_factors=None) -> pds_dims:
    """``pds_dims`` of any object with the model fields (n_layers, d_model,
    n_heads, n_kv_heads, head_dim, ffn_dim, rope_theta, rms_eps) and of an
    optional variant (rope_layout "neox"/"norm", rot_dim, rope_mscale,
    attn_softcap, window); ``freq_factors`` is a float32 array or None.  The
    returned struct keeps the factors' C array alive (``_keep``)."""
    pd = pds_dims(dims.n_layers, dims.d_model, dims.n_heads, dims.n_kv_heads, dims.head_dim,
                  dims.ffn_dim, dims.rope_theta, dims.rms_eps)
    if variant is not None:
        pd.rope_layout = PDS_ROPE_NORM if variant.rope_layout == "norm" else PDS_ROPE_NEOX
        pd.rot_dim = int(variant.rot_dim or 0)
        pd.rope_mscale = float(variant.rope_mscale or 0.0)
        pd.attn_softcap = float(variant.attn_softcap or 0.0)
        pd.window = int(variant.window or 0)
    if freq_factors is not None:
        arr = (ctypes.c_float * len(freq_factors))(*[float(f) for f in freq_factors])
        pd.freq_factors = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        pd._keep = arr
    return pd
