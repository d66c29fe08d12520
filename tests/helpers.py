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


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (2^(e - 7) for |x| in [2^e, 2^(e+1)))."""
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return np.exp2(e - 7)


def assert_close_block(x, ref, f_ref, o_ref, gate1, gate2, r_in, what="block"):
    """Whole-block FP32 output: the last two steps add gate * y for bf16
    hand-offs y = o, f, where a one-ulp rounding disagreement between two
    correct evaluations is expected; the elementwise bound is therefore
    2e-2 * max(1, |ref|) + |gate2| * ulp(f) + |gate1| * ulp(o), and the
    relative-L2 bound 1e-2 is unchanged. The same bounds apply to the
    residual increment out - r_in (gate1 * o + gate2 * f), which is small
    next to the residual and would hide a wrong gate."""
    x = np.asarray(x, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    r_in = np.asarray(r_in, np.float64).reshape(np.shape(ref))
    assert np.all(np.isfinite(x)), f"{what}: non-finite output"
    g1 = np.abs(np.asarray(gate1, np.float64))
    g2 = np.abs(np.asarray(gate2, np.float64))
    g1 = g1[None, :] if g1.ndim == 1 else g1
    g2 = g2[None, :] if g2.ndim == 1 else g2
    slack = g2 * bf16_ulp(f_ref) + g1 * bf16_ulp(o_ref)
    for name, a, b in (("output", x, ref), ("increment", x - r_in, ref - r_in)):
        bound = BF16_ELEM * np.maximum(1.0, np.abs(b)) + slack
        ratio = np.max(np.abs(a - b) / bound)
        r = rel_l2(a, b)
        assert ratio <= 1.0 and r <= BF16_REL_L2, \
            f"{what} {name}: max err/bound {ratio:.3g}, rel-L2 {r:.3g}"
