"""FreeSolo FS-L sparse attention forward, GB300-native (sm_103a).

The compute path lives in the C-ABI library built from ``csrc/`` (declared in
``include/fs.h``); ``long_context_lm_gb300.fs`` is its thin Python binding and
``long_context_lm_gb300.inputs`` the seeded synthetic input generator.
"""
__all__ = ["fs", "inputs"]
