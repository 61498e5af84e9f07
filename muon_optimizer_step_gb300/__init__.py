"""GB300-native sharded Muon optimizer step (sm_103a CUDA kernels behind a C ABI).

The compute lives in ``libmuon.so`` (built from ``csrc/``); ``muon_optimizer_step_gb300.capi``
is the ctypes binding with the same names as the C entry points.  Importing the binding
loads the library and raises if it is missing: there is no fallback path.
"""
