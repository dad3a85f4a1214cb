"""CPU oracle of the MoE layer forward (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never calls it and shares no code with
it: the oracle has its own bfloat16 conversion, its own top-k, its own
dispatch and its own FFN, all in float64 numpy (a BLAS matrix product is the
one library primitive it leans on).

What each function follows is stated in its docstring.  The pages describe
one engine ("Colibri", a C MoE inference engine) on five blog pages; they are
cited by host name, page title where the page has one, and section.
"""

from .moe import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    to_f64,
    round_to_bf16,
    router_logits,
    topk_select,
    softmax_selected,
    soft_route,
    dispatch,
    capacity_keep,
    silu,
    swiglu_expert,
    combine,
    moe_layer,
    token_outputs,
    rmsnorm,
    stack_layer,
    near_tie_tokens,
)
from .quant import (  # noqa: F401
    quantize_int8_block64,
    dequantize_int8_block64,
    quantize_experts,
    dequantize_experts,
)
