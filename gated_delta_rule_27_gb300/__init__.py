"""libkda: the Kimi Delta Attention (KDA) state recurrence on one GB300 (sm_103a).

The compute lives in libkda.so (C ABI, include/kda.h).  ``libkda`` is its
ctypes binding; ``workloads`` draws seeded synthetic inputs.
"""
__all__ = ["libkda", "workloads", "build"]
