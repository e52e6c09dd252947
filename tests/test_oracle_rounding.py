"""Pins of the oracle's rounding rules: Table 1 closed forms, unbiasedness,
brute-force nearest level, and the SR-versus-RTN error ordering.

The rules are those named by the listing page "Rounding in Preconditioner
Space", Table 1 (State-RTN, State-SR, Update-RTN, Update-SR); the closed forms
for the cell next to zero are read from tests/golden/table1_near_zero_cell.txt.
"""
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "table1_near_zero_cell.txt")


def _table1():
    rows = {}
    for line in open(GOLD):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            rows[k] = v
    return rows


def r_of(x, c2, eps):
    """Preconditioner 1/(sqrt(x)*c2 + eps) in float64 (closed form)."""
    return 1.0 / (np.sqrt(np.asarray(x, np.float64)) * c2 + eps)


def _near_zero_block(vt_over_b: float):
    """A Dyn4 block of scale 1 whose element 0 sits at vt = vt_over_b * b in the first cell."""
    L = O.codebooks()["dyn4"]
    b = float(L[1])
    x = np.zeros(2, np.float32)
    x[1] = 1.0            # sets the block scale s = 1
    x[0] = np.float32(vt_over_b * b)
    return L, O.codebooks()["dyn4_t"], x, b


def _mc_codes(L, t, x, rule, n_draws, c2=1.0, eps=1e-8, seed=5):
    """Codes of element 0 over n_draws independent draws (Philox stream, purpose 1)."""
    codes = np.empty(n_draws, np.uint8)
    w = O.draws(seed, 1, 0, 0, n_draws, 1)
    for i in range(n_draws):
        c, _ = O.quant_block(L, t, x, rule, words=np.array([w[i], 0], np.uint32), c2=c2, eps=eps)
        codes[i] = c[0]
    return codes


def test_table1_state_rtn_and_update_rtn_are_deterministic():
    tab = _table1()
    for frac in (0.01, 0.1, 0.3, 0.49):
        L, t, x, b = _near_zero_block(frac)
        c, s = O.quant_block(L, t, x, "state_rtn")
        assert s == 1.0
        assert float(c[0] == 0) == float(tab["state_rtn"])            # P(Q=0) = 1
        c, _ = O.quant_block(L, t, x, "update_rtn", c2=1.0, eps=1e-8)
        assert float(c[0] == 0) == float(tab["update_rtn"])           # P(Q=0) = 0


@pytest.mark.parametrize("frac", [0.05, 0.25, 0.45])
def test_table1_state_sr_probability(frac):
    assert _table1()["state_sr"] == "1-v/b"
    L, t, x, b = _near_zero_block(frac)
    n = 20000
    codes = _mc_codes(L, t, x, "state_sr", n)
    assert set(np.unique(codes)) <= {0, 1}
    p0 = (codes == 0).mean()
    p_exact = 1.0 - float(x[0]) / b
    assert abs(p0 - p_exact) < 4.5 * np.sqrt(p_exact * (1 - p_exact) / n)


@pytest.mark.parametrize("eps", [1e-3, 1e-4, 1e-5])
def test_table1_update_sr_probability_is_theta_eps(eps):
    assert _table1()["update_sr"] == "theta_eps"
    L, t, x, b = _near_zero_block(0.1)
    n = 60000
    codes = _mc_codes(L, t, x, "update_sr", n, c2=1.0, eps=eps)
    p0 = (codes == 0).mean()
    v = float(x[0])
    r_v, r_b, r_0 = r_of(v, 1.0, eps), r_of(b, 1.0, eps), 1.0 / eps
    p_exact = (r_v - r_b) / (r_0 - r_b)
    assert abs(p0 - p_exact) < 4.5 * np.sqrt(p_exact * (1 - p_exact) / n) + 1e-6
    # Theta(eps): p / eps tends to r(v) - r(b) evaluated at eps = 0
    lim = 1.0 / np.sqrt(v) - 1.0 / np.sqrt(b)
    assert 0.3 < p_exact / (eps * lim) < 1.7


def test_update_sr_is_unbiased_in_r_and_state_sr_in_v():
    rng = np.random.default_rng(3)
    L, t = O.codebooks()["dyn4"], O.codebooks()["dyn4_t"]
    # eps large enough that r(0) = 1/eps keeps P(Q=0) measurable by Monte Carlo
    c2, eps = 1.3, 1e-2
    x = np.minimum(np.abs(rng.normal(0, 0.5, 16)) ** 3, 1.9).astype(np.float32)
    x[0] = 2.0      # block scale
    x[1] = 2e-4     # inside the first cell (levels 0 and 0.001 * s)
    n = 40000
    w_all = O.draws(11, 1, 0, 0, n * 16, 1).reshape(n, 16)
    rs = np.zeros(16)
    vs = np.zeros(16)
    rs2 = np.zeros(16)
    vs2 = np.zeros(16)
    s = None
    for i in range(n):
        cu, s = O.quant_block(L, t, x, "update_sr", words=w_all[i], c2=c2, eps=eps)
        cs, _ = O.quant_block(L, t, x, "state_sr", words=w_all[i], c2=c2, eps=eps)
        rq = r_of(L[cu].astype(np.float64) * float(s), c2, eps)
        vq = L[cs].astype(np.float64) * float(s)
        rs += rq
        rs2 += rq * rq
        vs += vq
        vs2 += vq * vq
    mr, mv = rs / n, vs / n
    sr = np.sqrt(np.maximum(rs2 / n - mr ** 2, 0) / n)
    sv = np.sqrt(np.maximum(vs2 / n - mv ** 2, 0) / n)
    xr = r_of(x, c2, eps)
    assert np.all(np.abs(mr - xr) <= 4.5 * sr + 1e-5 * xr)
    assert np.all(np.abs(mv - x) <= 4.5 * sv + 1e-6 * x)


@pytest.mark.parametrize("name", ["nf4", "dyn4", "dyn4nz", "sdyn4", "lin4nz"])
def test_rtn_is_brute_force_nearest_level(name):
    rng = np.random.default_rng(1)
    L, t = O.codebooks()[name], O.codebooks()[name + "_t"]
    for trial in range(200):
        n = int(rng.integers(1, 129))
        x = rng.normal(0, 1, n).astype(np.float32) * np.float32(10.0 ** rng.uniform(-20, 20))
        if name not in ("nf4", "sdyn4"):
            x = np.abs(x)
        c, s = O.quant_block(L, t, x, "state_rtn")
        assert s == np.abs(x).max()
        a = L.astype(np.float64) * float(s)
        d = np.abs(x[:, None].astype(np.float64) - a[None, :])
        best = d.min(axis=1)
        got = d[np.arange(n), c]
        # nearest level, up to the FP32 rounding of the scaled thresholds
        assert np.all(got <= best * (1 + 1e-6) + 1e-6 * float(s))


def test_rtn_identity_on_levels():
    # quant o dequant is the identity on codebook levels (power-of-two scale: exact products)
    for name in ("nf4", "dyn4", "dyn4nz", "sdyn4", "lin4nz"):
        L, t = O.codebooks()[name], O.codebooks()[name + "_t"]
        for s in (1.0, 2.0 ** -20, 2.0 ** 30):
            x = (L * np.float32(s)).astype(np.float32)
            c, sc = O.quant_block(L, t, x, "state_rtn")
            assert sc == np.float32(s)
            assert np.array_equal(c, np.arange(16))
            # SR rules also keep exact levels
            for rule in ("state_sr", "update_sr"):
                w = O.draws(1, 1, 0, 0, 16, 1)
                c2, _ = O.quant_block(L, t, x, rule, words=w, c2=1.0, eps=1e-8)
                if name not in ("nf4", "sdyn4") or rule == "state_sr":
                    assert np.array_equal(c2, np.arange(16)), (name, rule)


def test_sr_error_dominates_rtn_error_pointwise():
    # Listing page Table 11 reports a larger relative RMS error for NF4-SR than
    # NF4-RTN; pointwise |x - Q_SR(x)| >= |x - Q_RTN(x)| implies that ordering.
    rng = np.random.default_rng(2)
    L, t = O.codebooks()["nf4"], O.codebooks()["nf4_t"]
    e_sr, e_rtn = [], []
    for trial in range(300):
        x = rng.normal(0, 1, 128).astype(np.float32)
        w = O.draws(7, trial + 1, 0, 0, 128, 0)
        cr, s = O.quant_block(L, t, x, "state_rtn")
        cs, _ = O.quant_block(L, t, x, "state_sr", words=w)
        qr = L[cr].astype(np.float64) * float(s)
        qs = L[cs].astype(np.float64) * float(s)
        er, es = np.abs(x - qr), np.abs(x - qs)
        assert np.all(es >= er - 1e-6 * float(s))
        e_sr.append(es)
        e_rtn.append(er)
    assert np.sqrt(np.mean(np.square(e_sr))) > np.sqrt(np.mean(np.square(e_rtn)))


def test_zero_block_codes():
    # s = 0: every RTN comparison is false (code 0); SR cells are the top level (15).
    for name in ("nf4", "dyn4", "dyn4nz"):
        L, t = O.codebooks()[name], O.codebooks()[name + "_t"]
        x = np.zeros(128, np.float32)
        c, s = O.quant_block(L, t, x, "state_rtn")
        assert s == 0 and np.all(c == 0)
        c, _ = O.quant_block(L, t, x, "update_sr", words=O.draws(1, 1, 0, 0, 128, 1))
        assert np.all(c == 15)
        c, _ = O.quant_block(L, t, x, "state_sr", words=O.draws(1, 1, 0, 0, 128, 1))
        assert np.all(c == 15)


def r_next(x, b2, c2n, eps):
    """Next-step zero-gradient preconditioner 1/(sqrt(b2 x) c2n + eps), float64."""
    return 1.0 / (np.sqrt(b2 * np.asarray(x, np.float64)) * c2n + eps)


def test_next_step_update_sr_is_unbiased_in_next_step_r():
    # the next-step variant of ZIP-SR: E[r'(Q)] = r'(v) for r' evaluated at
    # step t+1 with a zero gradient (beta2 = 0.8, step t = 2)
    rng = np.random.default_rng(4)
    L, t = O.codebooks()["dyn4"], O.codebooks()["dyn4_t"]
    b2, eps = 0.8, 1e-2
    c2n = float(np.float32(1.0 / np.sqrt(1.0 - b2 ** 3)))
    x = np.minimum(np.abs(rng.normal(0, 0.5, 16)) ** 3, 1.9).astype(np.float32)
    x[0] = 2.0
    x[1] = 2e-4
    n = 40000
    w_all = O.draws(12, 1, 0, 0, n * 16, 1).reshape(n, 16)
    rs = np.zeros(16)
    rs2 = np.zeros(16)
    for i in range(n):
        cu, s = O.quant_block(L, t, x, "update_sr", words=w_all[i], c2=c2n, eps=eps, rbeta=b2)
        rq = r_next(L[cu].astype(np.float64) * float(s), b2, c2n, eps)
        rs += rq
        rs2 += rq * rq
    mr = rs / n
    sr = np.sqrt(np.maximum(rs2 / n - mr ** 2, 0) / n)
    xr = r_next(x, b2, c2n, eps)
    assert np.all(np.abs(mr - xr) <= 4.5 * sr + 1e-5 * xr)


@pytest.mark.parametrize("eps", [1e-3, 1e-4])
def test_next_step_update_sr_near_zero_probability(eps):
    # Table 1's cell next to zero in the next-step space: P(Q=0) =
    # (r'(v) - r'(b)) / (r'(0) - r'(b)), still Theta(eps)
    L, t, x, b = _near_zero_block(0.1)
    b2, c2n = 0.9, 1.25
    n = 60000
    w = O.draws(5, 1, 0, 0, n, 1)
    codes = np.empty(n, np.uint8)
    for i in range(n):
        c, _ = O.quant_block(L, t, x, "update_sr", words=np.array([w[i], 0], np.uint32), c2=c2n, eps=eps,
                             rbeta=b2)
        codes[i] = c[0]
    p0 = (codes == 0).mean()
    v = float(x[0])
    r_v, r_b, r_0 = r_next(v, b2, c2n, eps), r_next(b, b2, c2n, eps), 1.0 / eps
    p_exact = (r_v - r_b) / (r_0 - r_b)
    assert abs(p0 - p_exact) < 4.5 * np.sqrt(p_exact * (1 - p_exact) / n) + 1e-6
    lim = (1.0 / np.sqrt(v) - 1.0 / np.sqrt(b)) / (np.sqrt(b2) * c2n)
    assert 0.3 < p_exact / (eps * lim) < 1.7
