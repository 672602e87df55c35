"""fp64 CPU oracle for the Event Tensor MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (``moe_layer_scheduling_gb300``)
never imports it and shares no code with it.
"""
from .oracle import *  # noqa: F401,F403
