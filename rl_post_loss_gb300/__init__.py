"""GB300-native fused GRPO + IcePop token-level policy loss (sm_103a).

The computation runs in the CUDA library ``librl_loss.so`` built from
``csrc/`` (C-ABI declared in ``include/rl_loss.h``); ``capi`` is the thin
ctypes binding over it and ``synthetic`` draws seeded inputs.
"""
__all__ = ["capi", "synthetic"]
