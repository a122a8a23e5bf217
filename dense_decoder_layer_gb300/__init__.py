"""GB300 (sm_103a) batched prefill through a run of dense Llama-style decoder layers.

``pds`` is the ctypes binding of the C ABI in ``include/pds.h`` (the
library ``libpds.so`` built by :mod:`.build`); ``stack.DenseStack`` owns
the PyTorch buffers of one stack.  Importing this package loads nothing;
the library is loaded on first use and must exist.
"""

__all__ = ["pds", "stack", "build"]
