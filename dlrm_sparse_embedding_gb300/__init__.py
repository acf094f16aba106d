"""GB300-native training step of a multi-table sparse embedding layer.

The compute lives in libemb.so (hand-written CUDA for sm_103a, C ABI in
include/emb.h); this package is a thin ctypes binding over it.  Importing the
package loads the library and fails if it has not been built.
"""
from ._lib import (EMB_ERR_CAPACITY, EMB_ERR_CUDA, EMB_ERR_INVALID_ARG, EMB_ERR_KEY_RANGE, EMB_ERR_OOM,
                   EMB_ERR_STATE, EMB_ERR_TIMEOUT, EMB_OK, EXPORTS, LIB_PATH, VARIANTS, EmbError, check, lib)
from .layer import EmbeddingLayer, unique, unique_workspace_bytes

__all__ = [
    "EmbeddingLayer", "unique", "unique_workspace_bytes", "EmbError", "check", "lib", "LIB_PATH", "EXPORTS",
    "VARIANTS", "EMB_OK", "EMB_ERR_INVALID_ARG", "EMB_ERR_OOM", "EMB_ERR_CUDA", "EMB_ERR_KEY_RANGE",
    "EMB_ERR_CAPACITY", "EMB_ERR_TIMEOUT", "EMB_ERR_STATE",
]
