"""GB300 (sm_103a) CSA2 index + sparse-attention decode step.

The compute path lives in the C-ABI library built from ``csrc/`` (see
``include/csa2.h``); ``abi`` is its ctypes binding, ``layer_group`` issues the
calls of one decoder layer group, ``workloads`` draws seeded synthetic inputs.
Importing this package does not load the library; importing ``abi`` does, and
fails loudly when it has not been built.
"""
__all__ = ["abi", "layer_group", "workloads", "build"]
