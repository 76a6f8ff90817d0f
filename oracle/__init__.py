"""Oracle of the routed + shared-expert MoE layer, forward and backward (test infrastructure).

A plain, slow, float64 CPU statement of the layer, written from the pages that
define the method.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU baseline / reference arm use it.  It shares no code with the
CUDA library, and the library never calls it.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
from . import moe_backward_oracle  # noqa: F401
from .moe_backward_oracle import dsilu, moe_backward, selected_weights_backward, swiglu_backward  # noqa: F401
