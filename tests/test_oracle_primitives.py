"""Pins of the oracle's primitives against things other than the oracle itself.

* Philox4x32-10 against cuRAND's host Philox4_32_10 generator (a library
  routine run on the CPU; no GPU needed).
* NF4 against the same construction through scipy.special.ndtri.
* Dyn4 / Dyn4-NZ against the exact rational definition.
* BF16 rounding against torch's float32 -> bfloat16 conversion.
* Host scalars against direct float64 evaluation.
"""
import ctypes
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O

CURAND = "/usr/local/cuda/lib64/libcurand.so"


def _curand_host_philox(seed: int, n: int) -> np.ndarray:
    lib = ctypes.CDLL(CURAND)
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return out
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.skipif(not os.path.exists(CURAND), reason="cuRAND not installed")
@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host_generator(seed):
    # cuRAND's host Philox generator emits, at offset 0, group j of four words
    # = Philox4x32-10(counter=(0, 0, j, 0), key=(seed_lo, seed_hi)).
    n = 4 * 4096
    ref = _curand_host_philox(seed, n)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for j in list(range(64)) + [1000, 2047, 4095]:
        got = O.philox([0, 0, j, 0], key)
        assert got.tolist() == ref[4 * j:4 * j + 4].tolist(), j


def test_draw_counter_layout():
    # Element idx uses word idx&3 of the call with counter (idx>>2, (idx>>34)|p<<28, tensor, step).
    seed, step, tid = 0x1234_5678_9ABC_DEF0, 7, 3
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for idx in [0, 1, 2, 3, 4, 1023, (1 << 34) + 5, (1 << 40) + 2]:
        for p in (0, 1):
            w = O.draws(seed, step, tid, idx, 1, p)[0]
            ctr = [(idx >> 2) & 0xFFFFFFFF, ((idx >> 34) | (p << 28)) & 0xFFFFFFFF, tid, step]
            assert w == O.philox(ctr, key)[idx & 3]
    # purposes, tensors and steps give different streams
    a = O.draws(seed, 1, 0, 0, 256, 0)
    assert (a != O.draws(seed, 1, 0, 0, 256, 1)).mean() > 0.99
    assert (a != O.draws(seed, 1, 1, 0, 256, 0)).mean() > 0.99
    assert (a != O.draws(seed, 2, 0, 0, 256, 0)).mean() > 0.99


def test_uniform_is_exact_24bit():
    w = np.array([0, 255, 256, 0xFFFFFFFF, 0x80000000, 0x12345678], dtype=np.uint32)
    for x in w:
        u = O.lib().oracle_uniform(int(x))
        assert u == (int(x) >> 8) / 2 ** 24
    assert O.lib().oracle_uniform(0xFFFFFFFF) < 1.0


def test_uniform_distribution():
    w = O.draws(99, 1, 0, 0, 200_000, 1)
    u = O.uniform(w).astype(np.float64)
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / u.size)
    hist, _ = np.histogram(u, bins=16, range=(0, 1))
    exp = u.size / 16
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 40  # 15 dof, p ~ 5e-4


def test_nf4_matches_scipy_construction():
    from scipy.special import ndtri
    d = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = [ndtri(d + i * ((0.5 - d) / 8.0)) for i in range(8)]
    neg = [-ndtri(d + i * ((0.5 - d) / 7.0)) for i in range(7)]
    vals = sorted(pos + neg + [0.0])
    ref = (np.array(vals) / max(vals)).astype(np.float32)
    nf4 = O.codebooks()["nf4"]
    assert np.array_equal(ref.view(np.uint32), nf4.view(np.uint32))


def test_nf4_structure():
    nf4 = O.codebooks()["nf4"]
    assert nf4.dtype == np.float32 and nf4.size == 16
    assert np.all(np.diff(nf4) > 0)
    assert nf4[0] == -1.0 and nf4[7] == 0.0 and nf4[15] == 1.0
    assert (nf4 < 0).sum() == 7 and (nf4 > 0).sum() == 8


def _nearest_f32(q: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational, checked against its float32 neighbours."""
    c = np.float32(float(q))
    cands = [c]
    lo = hi = c
    for _ in range(2):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        cands += [lo, hi]
    best = min(cands, key=lambda x: (abs(Fraction(float(x)) - q), int(np.array(x).view(np.uint32)) & 1))
    return best


@pytest.mark.parametrize("nz", [False, True])
def test_dyn4_exact_rationals(nz):
    lv = O.codebooks()["dyn4nz" if nz else "dyn4"]
    exact = [Fraction(1, 10 ** 4) if nz else Fraction(0)]
    for e in range(4):
        f = 3 - e
        for j in range(2 ** f):
            exact.append(Fraction(2 ** f + 9 * (j + 1), 10 ** (e + 1) * 2 ** f))
    exact.sort()
    for x, q in zip(lv, exact):
        assert x == _nearest_f32(q), (x, q)
    assert np.all(np.diff(lv) > 0) and lv[-1] == 1.0
    if nz:
        assert lv.min() > 0
    else:
        assert lv[0] == 0.0


def test_sdyn4_exact_rationals():
    # signed dynamic-exponent map: rung i = 0..2 splits [1/10, 1] into 2^i equal
    # parts; their midpoints times 10^(i-2), with both signs, plus 0 and +1
    lv = O.codebooks()["sdyn4"]
    mags = []
    for i in range(3):
        for j in range(2 ** i):
            mid = Fraction(1, 10) + Fraction(9 * (2 * j + 1), 20 * 2 ** i)
            mags.append(mid * Fraction(10) ** (i - 2))
    exact = sorted(mags + [-m for m in mags] + [Fraction(0), Fraction(1)])
    assert len(exact) == 16
    for x, q in zip(lv, exact):
        assert x == _nearest_f32(q), (x, q)
    assert np.all(np.diff(lv) > 0) and lv[-1] == 1.0 and 0.0 in lv
    # symmetric except the top level
    assert sorted((-lv[lv != 1.0]).tolist()) == sorted(lv[lv != 1.0].tolist())


def test_lin4nz_exact_rationals():
    lv = O.codebooks()["lin4nz"]
    assert [Fraction(float(x)) for x in lv] == [Fraction(k, 16) for k in range(1, 17)]
    assert lv.min() > 0


def test_thresholds_are_rounded_midpoints():
    cb = O.codebooks()
    for name in ("nf4", "dyn4", "dyn4nz", "sdyn4", "lin4nz"):
        L, t = cb[name], cb[name + "_t"]
        assert t.size == 15
        for k in range(15):
            mid = (Fraction(float(L[k])) + Fraction(float(L[k + 1]))) / 2
            assert t[k] == _nearest_f32(mid)
            assert L[k] < t[k] < L[k + 1]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 1000), [0.0, -0.0, 1e38, -3.3895e38]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_round(x), ref)


@pytest.mark.parametrize("t", [1, 2, 10, 9001])
def test_host_scalars(t):
    lr, b1, b2, wd = np.float32(1e-3), np.float32(0.9), np.float32(0.999), np.float32(0.1)
    h = O.host_scalars(lr, b1, b2, wd, t)
    d1, d2, dl, dw = float(b1), float(b2), float(lr), float(wd)
    assert h["c2"] == np.float32(1 / np.sqrt(1 - d2 ** t))
    assert h["step_size"] == np.float32(dl / (1 - d1 ** t))
    assert h["decay"] == np.float32(1 - dl * dw)
    assert h["omb1"] == np.float32(1 - d1) and h["omb2"] == np.float32(1 - d2)
