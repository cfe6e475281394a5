"""DMuon owner-side Muon step on GB300 (sm_103a).

The compute path lives in the C-ABI library ``libdmuon.so`` (CUDA kernels for
sm_103a, declared in ``include/dmuon.h``); :mod:`newton_schulz_owner_gb300.dmuon`
is its thin ctypes binding.  Importing this package loads nothing: the binding
loads the library on first import and raises if it has not been built.
"""
__all__ = ["dmuon", "workloads"]
