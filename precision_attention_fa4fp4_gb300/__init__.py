"""Block-scaled FP4 FlashAttention with Direct-P for GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (``include/fa4fp4.h``); the
functions exported here only marshal torch tensors to that library.  Importing
the package does not load the library; the first call does, and raises if the
built library is missing.  There is no CPU fallback.
"""
from .inputs import Workload, make_inputs  # noqa: F401  (no CUDA needed)

_API = ("quantize", "fwd", "bwd", "bf16_fwd", "qtensor_alloc", "sync_status", "library_path",
        "load_library", "FMT_MXFP4", "FMT_MXFP8", "ALONG_D", "ALONG_N", "OUT_F32", "OUT_BF16",
        "QTensor", "Fa4Fp4Error")


def __getattr__(name):
    if name in _API:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
