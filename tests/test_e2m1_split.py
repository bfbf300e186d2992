"""The e2m1 term split the decode expert kernels apply to activations,
restated in numpy from its description and held to the accuracy the design
relies on.  Each 32-element group is carried as kFp4Terms e2m1 terms q_t
with their own UE8M0 scale 2^S_t: S_t is the smallest exponent that puts
the group's largest remaining magnitude at or below 6 (the largest e2m1
value), q_t = RN_e2m1(r_t 2^-S_t) (ties to even, saturating), r_{t+1} =
r_t - q_t 2^S_t.  (The e2m1 grid and rounding are the OCP MX ones the
MXFP4 weights use: kimi-k3-mlx README, "Tiers".)

What is pinned: the scale rule (every scaled group fits e2m1), the
worst-case shrink of a group's residual per term (a factor 3: the scaled
maximum lies in (3, 6] and a residual is at most half the local e2m1 step,
at most 1), and the measured accuracy of six terms on bf16 inputs of the
three shapes the layer feeds the split (Gaussian latents, heavy tails,
SiTU-GLU outputs), against four terms, which the per-step checks of the
GPU tests reject."""
import numpy as np
import pytest

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
TERMS = 6  # kFp4Terms of the decode kernels


def rn_e2m1(v: np.ndarray) -> np.ndarray:
    a, s = np.abs(v), np.sign(v)
    lo = np.clip(np.searchsorted(E2M1, a, side="right") - 1, 0, 7)
    hi = np.clip(lo + 1, 0, 7)
    dlo, dhi = a - E2M1[lo], E2M1[hi] - a
    tie_even = np.where(lo % 2 == 0, E2M1[lo], E2M1[hi])
    out = np.where(dlo < dhi, E2M1[lo], np.where(dhi < dlo, E2M1[hi], tie_even))
    return s * np.where(a >= 6.0, 6.0, out)


def scale_exponent(m: np.ndarray) -> np.ndarray:
    """Smallest S with m * 2^-S <= 6, for m = mant * 2^e, mant in [1, 2)."""
    f, e = np.frexp(m)
    mant, ee = 2.0 * f, e - 1
    s = ee - 2 + (mant > 1.5)
    return np.where(m == 0, -127, np.maximum(s, -127))


def split(x: np.ndarray, n: int):
    r = x.reshape(-1, 32).astype(np.float64)
    x0 = r.copy()
    maxima = []
    for _ in range(n):
        m = np.abs(r).max(axis=1, keepdims=True)
        maxima.append(m)
        sc = np.ldexp(1.0, scale_exponent(m))
        assert np.all(m / sc <= 6.0)
        assert np.all((m == 0) | (m / sc > 3.0) | (sc == np.ldexp(1.0, -127)))
        r = r - rn_e2m1(r / sc) * sc
    return x0, r, maxima


def bf16(v: np.ndarray) -> np.ndarray:
    u = v.astype(np.float32).view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.view(np.float32).astype(np.float64)


def inputs(seed: int, n: int = 1 << 18):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal(n)
    return {"gauss": bf16(g), "t3": bf16(rng.standard_t(3, n)),
            "situ": bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(rng.standard_normal(n) / 25))}


@pytest.mark.parametrize("name", ["gauss", "t3", "situ"])
def test_six_terms_accuracy(name):
    x = inputs(11)[name]
    x0, r, maxima = split(x, TERMS)
    gmax = np.abs(x0).max(axis=1, keepdims=True)
    # worst case: each term shrinks the group's largest residual at least 3x
    for a, b in zip(maxima, maxima[1:] + [np.abs(r).max(axis=1, keepdims=True)]):
        assert np.all(b <= a / 3.0 + 1e-300)
    assert np.all(np.abs(r) <= gmax * 3.0 ** -TERMS)
    # measured: far inside that bound
    rel_rms = np.sqrt(np.mean(r ** 2) / np.mean(x0 ** 2))
    assert rel_rms < 2e-7, rel_rms
    assert np.max(np.abs(r) / np.maximum(gmax, 1e-300)) < 4e-6


def test_four_terms_are_not_enough():
    """Four terms leave ~1e-4 of the activation: above the 2e-5 the o check
    of the GPU tests allows for the product of the GPU's own h."""
    x = inputs(12)["t3"]
    x0, r, _ = split(x, 4)
    assert np.sqrt(np.mean(r ** 2) / np.mean(x0 ** 2)) > 2e-5


def test_exact_cases():
    """Values on the e2m1 grid of their group's scale come back exactly in
    one term; zero groups stay zero."""
    rng = np.random.default_rng(5)
    codes = rng.choice(np.concatenate([E2M1, -E2M1]), size=(64, 32))
    codes[:, 0] = 6.0  # fixes the scale at 2^0 for every group
    x0, r, _ = split(codes.reshape(-1) * 1.0, 1)
    assert np.all(r == 0)
    x0, r, _ = split(np.zeros(64), TERMS)
    assert np.all(r == 0)
