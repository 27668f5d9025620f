"""GB300-native single-GPU MoE layer forward (sm_103a CUDA behind a C ABI).

The compute path is the CUDA library ``libmoe.so`` built from ``csrc/``; the
functions of ``router_experts_gb300.moe`` marshal torch tensors into its C
entry points.  There is no CPU or PyTorch fallback: if the library is missing,
every call raises.
"""
__all__ = ["workloads"]
