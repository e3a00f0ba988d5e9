"""fp64 CPU oracle of the MoE expert layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg
of ``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or runs anything here, and this
package shares no code with it: only the seeded input generators in
``synth`` (which hold none of the method's arithmetic) serve both sides.

Pins: every function is checked by ``tests/test_oracle_pins.py`` against
something other than itself (worked examples printed on the pages, closed
forms, library routines on special cases, finite differences, brute force).
The token-rounding tie rules (half-up rounding, score ties broken by token
index) are readings of a rule the pages state only in words; the brute-force
pin checks the oracle against that reading, not against the pages' own
(absent) algorithm listing.
"""
from .moe_oracle import (  # noqa: F401
    Routing,
    bf16_bits_to_f64,
    capacity_drop,
    combine,
    combine_weights,
    dequantize_blocks_mx,
    dequantize_rows_e4m3,
    dequantize_token_blocks_mx,
    e4m3_decode,
    e4m3_encode,
    e4m3_round,
    expert_block_backward,
    expert_capacity,
    expert_ffn,
    group_by_expert,
    moe_backward,
    moe_forward,
    moe_forward_fp8,
    moe_forward_mx,
    mx_block_exponents,
    round_bf16,
    route_discrete,
    router_logits,
    quantize_blocks_mx,
    quantize_rows_e4m3,
    softmax,
    token_rounding,
    topk_experts,
)
from .metrics import WEIGHT_GRAD, compare, rel_error  # noqa: F401
