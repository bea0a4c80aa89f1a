"""GB300 (sm_103a) CCA prefill: global-aware pooling and fused core/local attention.

The compute runs in the CUDA library ``libcca.so`` behind a C ABI
(``include/cca.h``); :mod:`.api` is a thin ctypes binding over it.  Importing
this package does not load the library; the first call does, and fails loudly
if it is missing.
"""
from .workloads import Workload  # noqa: F401

__all__ = ["Workload"]
