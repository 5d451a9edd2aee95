"""B300-native MoE layer forward pass: TopK-then-softmax routing, capacity-limited
dispatch, grouped expert FFN on tcgen05 tensor cores, fixed-order combine and the
load-balancing loss.

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/moe.h``); ``top_routing_expert_then_b300.lib`` is the thin
ctypes binding. Importing this package does not load the library.
"""

__all__ = ["inputs", "lib"]
