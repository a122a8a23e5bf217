"""CPU fp64 oracle of the dense decoder-layer prefill stack.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path
(the C-ABI library and its Python binding) never calls it, and this
package imports nothing from the product.

Every function is the plain definition of one step, in float64, with a
library matmul as the only primitive; see :mod:`oracle.stack`.
"""

from .stack import (  # noqa: F401
    widen_bf16,
    rms_norm,
    rope_inv_freq,
    rope_neox,
    rope_rotate,
    silu,
    causal_gqa_attention,
    decoder_layer,
    prefill_dense_stack,
)
