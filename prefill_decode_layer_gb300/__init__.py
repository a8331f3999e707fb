"""GB300 (sm_103a) implementation of the ds4 per-token layer step, layer-major
prefill, lm_head and sampler, behind the C ABI declared in include/ds4g.h.

Python only marshals arguments to the native library (``libds4g.so``); every step
of the computation runs in its CUDA kernels.  Importing the binding fails loudly
if the library has not been built.
"""
from .ds4g import (BF16, DEBUG, F32, Ds4gError, Model, Session, config_struct, lib,  # noqa: F401
                   sample, sample_static, sample_u, sample_workspace_bytes, session_bytes)
