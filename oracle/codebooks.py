"""Codebooks of the oracle, built from their published definitions.

TEST INFRASTRUCTURE ONLY (see oracle/oracle.py).  The CUDA library builds its
own copies with a different method; the two are compared bit for bit by the
tests, never shared.

The pages name the codebooks but print no levels:
  * NF4 for the first moment -- "Rounding in Preconditioner Space" listing
    page, Abstract and Table 2; news page paragraph 3.
  * Dyn4 (zero-inclusive dynamic exponent) for v under ZIP-SR and Dyn4-NZ
    (zero-excluding) under ZE-EDEN -- listing page Table 2, Figure 1 caption;
    AReno docs "State representation" ("excludes zero").

Readings (the pages are silent on the level values):
  * NF4 follows the 4-bit NormalFloat construction of Dettmers et al.
    (QLoRA, 2023): with delta = 1 - (1/30 + 1/32)/2, positives are
    Phi^-1 of 8 evenly spaced probabilities from delta towards 0.5 (the 0.5
    end excluded), negatives are -Phi^-1 of 7 such points, plus one exact
    zero; everything is divided by the largest value.  Computed in double,
    rounded once to FP32.  Phi^-1 here is statistics.NormalDist.inv_cdf.
  * Dyn4 is the unsigned 4-bit dynamic-exponent map (dynamic tree
    quantisation, Dettmers et al.): a code with e leading zero bits
    (e = 0..3) is followed by an indicator 1 and f = 3 - e fraction bits
    and decodes to 10^-e * (0.1 + 0.9 * (j + 1) / 2^f), j < 2^f; the
    all-zero code is 0.  Dyn4-NZ maps the all-zero code to the next
    exponent rung, 10^-4, so no level is zero.
  * SDyn4 (TorchAO baseline's first moment, listing page Table 2) is the
    signed 4-bit dynamic-exponent map as the dynamic quantisation of
    Dettmers et al. defines it for 4 bits with 3 exponent rungs: on rung
    i = 0, 1, 2 the interval [0.1, 1] is cut into 2^i equal parts whose
    midpoints, scaled by 10^(i-2), are the magnitudes (7 in all); both
    signs of each, plus 0 and +1, give 16 levels.
  * Lin4-NZ (TorchAO baseline's second moment, Table 2) is the linear
    zero-excluding map k/16, k = 1..16.
  * Codes index the levels sorted ascending.  RTN thresholds are the FP32
    rounding of the double midpoint of adjacent FP32 levels.
"""
from statistics import NormalDist

import numpy as np


def nf4_levels() -> np.ndarray:
    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    inv = NormalDist().inv_cdf
    pos = [inv(delta + i * ((0.5 - delta) / 8.0)) for i in range(8)]
    neg = [-inv(delta + i * ((0.5 - delta) / 7.0)) for i in range(7)]
    vals = sorted(pos + neg + [0.0])
    top = max(vals)
    return np.array([v / top for v in vals], dtype=np.float64).astype(np.float32)


def dyn4_levels(zero_excluding: bool = False) -> np.ndarray:
    vals = []
    for e in range(4):
        f = 3 - e
        for j in range(2 ** f):
            vals.append(10.0 ** (-e) * (0.1 + 0.9 * (j + 1) / 2 ** f))
    vals.append(1e-4 if zero_excluding else 0.0)
    return np.array(sorted(vals), dtype=np.float64).astype(np.float32)


def sdyn4_levels() -> np.ndarray:
    mags = []
    for i in range(3):
        parts = 2 ** i
        for j in range(parts):
            lo = 0.1 + 0.9 * j / parts
            hi = 0.1 + 0.9 * (j + 1) / parts
            mags.append(10.0 ** (i - 2) * (lo + hi) / 2.0)
    vals = sorted([m for m in mags] + [-m for m in mags] + [0.0, 1.0])
    return np.array(vals, dtype=np.float64).astype(np.float32)


def lin4nz_levels() -> np.ndarray:
    return np.array([k / 16.0 for k in range(1, 17)], dtype=np.float64).astype(np.float32)


def midpoints(levels: np.ndarray) -> np.ndarray:
    lv = levels.astype(np.float64)
    return ((lv[:-1] + lv[1:]) / 2.0).astype(np.float32)


def all_codebooks() -> dict:
    nf4 = nf4_levels()
    d4 = dyn4_levels(False)
    d4nz = dyn4_levels(True)
    sd4 = sdyn4_levels()
    l4 = lin4nz_levels()
    return {
        "nf4": nf4, "nf4_t": midpoints(nf4),
        "dyn4": d4, "dyn4_t": midpoints(d4),
        "dyn4nz": d4nz, "dyn4nz_t": midpoints(d4nz),
        "sdyn4": sd4, "sdyn4_t": midpoints(sd4),
        "lin4nz": l4, "lin4nz_t": midpoints(l4),
    }
