"""Prefix-reused suffix prefill on one GB300 (sm_103a).

The compute path is libkvr.so (hand-written CUDA behind a C ABI, declared in
include/kvr.h); ``kvr`` is a thin ctypes binding with the same names.  There
is no CPU fallback: importing the binding without the built library raises.
"""
from .kvr import (KVR_OK, KvrError, Kvr, config_for_shape, layer_weight_structs,  # noqa: F401
                  load_library)
