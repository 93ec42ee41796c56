"""GB300-native (sm_103a) absorbed-form MLA decode / causal speculative verify.

The compute path is a C-ABI shared library of hand-written CUDA kernels
(``csrc/``, declared in ``include/mla_gb300.h``); ``mla`` is its thin ctypes
binding and ``workloads`` draws the seeded synthetic inputs.
"""
__version__ = "0.1.0"
