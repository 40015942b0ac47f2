"""GB300-native block-cached, confidence-threshold masked-diffusion decoding.

The compute path is the C-ABI library ``libdllm.so`` (hand-written sm_103a CUDA
kernels) declared in ``include/dllm.h``; ``binding`` is its thin ctypes layer.
Importing this package loads nothing: the library is opened on first use and
raises if it has not been built.
"""
from .configs import MODELS, WORKLOADS, ModelConfig, Workload  # noqa: F401
