"""GB300-native continuous-batching decode step.

The hot path lives in ``libcbt.so`` (hand-written sm_103a CUDA kernels behind the C ABI
of ``include/cbt.h``); ``binding`` mirrors that ABI under the same names, and ``model``
lays out synthetic weights and owns engine handles.  There is no CPU or PyTorch
fallback: if the library is not built, every call raises.
"""
from . import binding  # noqa: F401
from ._build import build  # noqa: F401
