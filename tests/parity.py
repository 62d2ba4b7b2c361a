"""Comparison helpers shared by the GPU parity tests (no arithmetic of the method)."""
import numpy as np


def row_gate(gpu: np.ndarray, ref: np.ndarray, strict: float = 2e-3):
    """Per-row gates against the float64 oracle.

    contract: max|gpu - ref| <= 1e-2 * max(1, rms(ref row))  (the stated bar)
    strict:   max|gpu - ref| <= strict * rms(ref row)          (fp32-arithmetic bar)
    Returns (worst contract ratio, worst strict ratio); both must be <= 1.
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU output"
    err = np.abs(gpu - ref).max(axis=1)
    rms = np.sqrt((ref ** 2).mean(axis=1))
    contract = err / (1e-2 * np.maximum(1.0, rms))
    strict_r = err / (strict * np.maximum(rms, 1e-300))
    return float(contract.max()), float(strict_r.max())


def assert_rows_close(gpu, ref, strict: float = 2e-3, what: str = ""):
    c, s = row_gate(gpu, ref, strict)
    assert c <= 1.0, f"{what}: contract gate exceeded ({c:.3g} x tolerance)"
    assert s <= 1.0, f"{what}: strict gate exceeded ({s:.3g} x tolerance)"


def sample_rows(M: int, n: int = 256, seed: int = 0) -> np.ndarray:
    """Deterministic sample: first row, last row and a seeded choice in between."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], mid]))
