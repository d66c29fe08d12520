"""Shared test helpers: tolerances and tensor conversion (no method arithmetic)."""
import numpy as np
import torch

# Tolerances for bf16 outputs: elementwise |gpu - ref| <= 2e-2 * max(1, |ref|)
# (max-abs 2e-2 measured in units of the value once it exceeds 1, because a
# bf16 ulp is already 3e-2 at magnitude 4) and relative L2 <= 1e-2. FP32
# residual outputs of the modulation step: relative L2 <= 1e-5.
BF16_ELEM = 2e-2
BF16_REL_L2 = 1e-2
F32_REL_L2 = 1e-5


def np64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, ref) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


def assert_close_bf16(x, ref, what=""):
    x = np.asarray(x, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x)), f"{what}: non-finite output"
    ratio = np.max(np.abs(x - ref) / (BF16_ELEM * np.maximum(1.0, np.abs(ref))))
    r = rel_l2(x, ref)
    assert ratio <= 1.0 and r <= BF16_REL_L2, f"{what}: max err/bound {ratio:.3g}, rel-L2 {r:.3g}"


def assert_close_f32(x, ref, what=""):
    r = rel_l2(np.asarray(x, np.float64), np.asarray(ref, np.float64))
    assert r <= F32_REL_L2, f"{what}: rel-L2 {r:.3g}"


def sample_rows(L: int, n: int, seed: int) -> np.ndarray:
    """Seeded row sample that always contains the first and the last valid row."""
    g = np.random.default_rng(seed)
    rows = g.choice(L, size=min(n, L), replace=False)
    rows[0], rows[-1] = 0, L - 1
    return np.unique(rows)
