"""Block-scaled FP4 FlashAttention with Direct-P for GB300 (sm_103a).

The compute lives in a C-ABI CUDA library (``include/fa4fp4.h``); the
functions exported here only marshal torch tensors to that library.  Importing
the package does not load the library; the first call does, and raises if the
built library is missing.  There is no CPU fallback.
"""
from .inputs import Workload, make_inputs  # noqa: F401  (no CUDA needed)

def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    import importlib
    api = importlib.import_module(__name__ + ".api")
    try:
        return getattr(api, name)
    except AttributeError:
        raise AttributeError(name) from None
