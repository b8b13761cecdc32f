"""Test infrastructure: the CPU oracle of the MoE layer (see moe_oracle).

Only tests, the smoke check and the bench's CPU-baseline legs import this
package; the library never does.
"""
from .moe_oracle import (dispatch, forward, backward, forward_rows, backward_rows,  # noqa: F401
                         weight_grad_slices, rel_err, check_distinct, silu, silu_grad,
                         sigmoid, expert_forward)
