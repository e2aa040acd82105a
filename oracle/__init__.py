"""CPU oracle for the MoE token-dispatch layer (test infrastructure only).

The oracle is a plain C library (``moe_oracle.c``) wrapped here with ctypes.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference arms of ``bench.py`` may import this package.  The product path
(``grouped_expert_gemm_moe_gb300``) never imports it.
"""
from .oracle import (  # noqa: F401
    build,
    load,
    route,
    permute,
    permute_capped,
    expert_hidden,
    expert_down,
    moe_layer,
    moe_layer_w8,
    quantize_w8,
    router_logits,
    num_threads,
)
