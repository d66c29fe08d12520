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
    report = {}
    for name, a, b in (("output", x, ref), ("increment", x - r_in, ref - r_in)):
        plain = BF16_ELEM * np.maximum(1.0, np.abs(b))
        err = np.abs(a - b)
        ratio = float(np.max(err / (plain + slack)))
        r = rel_l2(a, b)
        # the same error against the bound without the hand-off slack: above
        # 1 where the slack is what admits a correct result
        report[name] = dict(ratio=ratio, ratio_without_slack=float(np.max(err / plain)),
                            rel_l2=r)
        assert ratio <= 1.0 and r <= BF16_REL_L2, \
            f"{what} {name}: max err/bound {ratio:.3g}, rel-L2 {r:.3g}"
    print(f"{what}: " + "; ".join(
        f"{k} max err/bound {v['ratio']:.3g} (without the hand-off slack "
        f"{v['ratio_without_slack']:.3g}), rel-L2 {v['rel_l2']:.3g}" for k, v in report.items()))
    return report


def assert_close_sage(x, ref, terms, L, what="sage attention"):
    """FP8 attention output against the oracle's: the two quantise every
    softmax weight p to E4M3 at different scales (the oracle as 448 p against
    the exact row maximum, the kernel as lambda * 448 p with lambda in
    (1/4, 1] from its integer running maximum), so each weight's code differs
    by up to half an E4M3 step on each side. terms = (a1, a0, v2, u2) from
    oracle.sage_error_terms. Checked:
      worst case, per element:  |x - ref| <= B + 2^-8 (|ref| + B),
        B = (2^-3 + 2^-15 + L 2^-23) a1 + (2^-10 + 2^-8) / 448 a0
        (half steps of 2^-4 p in E4M3's normal range, below it 2^-10 / 448
        and 2^-10 / (448 lambda) < 2^-8 / 448; exp2 and score rounding
        2^-15; FP32 accumulation of P V; the two bf16 output roundings);
      in the mean: sum (x - ref)^2 <= 4 * sum E[(x - ref)^2], with
        E[(x - ref)^2] <= (2/3) 2^-8 v2 + ((2^-10)^2 + (2^-8)^2) / (3 448^2) u2
                          + (2/3) 2^-18 ref^2
        (two independent roundings, each uniform within its half step)."""
    x = np.asarray(x, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    a1, a0, v2, u2 = (np.asarray(t, np.float64).reshape(ref.shape) for t in terms)
    assert np.all(np.isfinite(x)), f"{what}: non-finite output"
    b = (2.0 ** -3 + 2.0 ** -15 + L * 2.0 ** -23) * a1 + (2.0 ** -10 + 2.0 ** -8) / 448.0 * a0
    bound = b + 2.0 ** -8 * (np.abs(ref) + b)
    err = x - ref
    worst = float(np.max(np.abs(err) / bound))
    expect = ((2.0 / 3.0) * 2.0 ** -8 * v2 + (2.0 ** -20 + 2.0 ** -16) / (3 * 448.0 ** 2) * u2
              + (2.0 / 3.0) * 2.0 ** -18 * ref * ref)
    mean_ratio = float(np.sum(err * err) / (4.0 * np.sum(expect)))
    assert worst <= 1.0 and mean_ratio <= 1.0, \
        f"{what}: worst-case ratio {worst:.3g}, mean-square ratio {mean_ratio:.3g}"
    return worst, mean_ratio
