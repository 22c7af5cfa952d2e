"""Helpers shared by the GPU tests (not collected: no test_ prefix)."""
import numpy as np

import oracle

# Tolerances for floating-point results against the fp64 oracle:
# relative Frobenius error and per-element |delta| <= ATOL_SCALE*(|ref|+1).
REL_FRO = 5e-3
ATOL_SCALE = 1e-2


def check_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    d = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    assert rel <= REL_FRO, "%s: relative Frobenius error %.3e" % (what, rel)
    bad = np.abs(d) > ATOL_SCALE * (np.abs(ref) + 1.0)
    assert not bad.any(), "%s: %d elements out of bound, worst at %s" % (
        what, int(bad.sum()), np.unravel_index(np.argmax(np.abs(d) - ATOL_SCALE * (np.abs(ref) + 1)), d.shape))
    return rel


def bf16(bits):
    return oracle.bf16_to_f64(bits)


def sample_rows(n: int, k: int, seed: int = 7) -> np.ndarray:
    """k distinct rows of n, always including the first and the last."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], mid]))
