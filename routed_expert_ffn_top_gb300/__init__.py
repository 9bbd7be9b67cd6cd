"""GB300-native (sm_103a) small-batch MoE decode block.

The compute lives in one C-ABI shared library built from ``csrc/`` (declared in
``include/moe.h``); :mod:`routed_expert_ffn_top_gb300.moe` is the thin ctypes binding with
the same entry-point names.  Importing this package does not load the library; the first
call into :mod:`.moe` does, and fails loudly if it has not been built.
"""

__all__ = ["moe", "synthetic"]
