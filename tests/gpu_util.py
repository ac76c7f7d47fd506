"""Helpers shared by the GPU parity tests (no arithmetic of the method)."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import precision_attention_fa4fp4_gb300 as fa
    fa.load_library()     # raises if the CUDA library is missing: no fallback
    return fa


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def round_like(x: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Round an FP64 reference to the output dtype of the kernel (bf16 via
    torch's round-to-nearest-even, else FP32)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    t = t.to(torch.bfloat16) if out_bf16 else t.to(torch.float32)
    return t.to(torch.float64).numpy()


# Parity bar for outputs and gradients (relative L2 and max-abs, after the
# oracle's result is rounded to the kernel's output dtype).
REL_L2_TOL = 1e-3
MAX_ABS_TOL = 1e-2


def assert_close(got, want, what, rel=REL_L2_TOL, mabs=MAX_ABS_TOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    r = rel_l2(got, want)
    m = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert r <= rel and m <= mabs, f"{what}: rel-L2 {r:.3g} (tol {rel}), max-abs {m:.3g} (tol {mabs})"
