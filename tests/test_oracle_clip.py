"""Pins of the oracle's global gradient-norm clipping.

AReno docs "4-bit AdamW", section "State representation": gradient norm and
clipping run directly on the BF16 gradient shards.  Reading (torch's
clip_grad_norm_ with the 2-norm): clip = min(1, max_norm * (1 / (||g|| + 1e-6)))
in FP32 (torch divides a scalar by a tensor as a reciprocal and a product),
multiplied into each FP32 gradient inside the step.

What pins it, independently of the oracle's own code:
  * the canonical sum of squares equals textbook recursive pairwise summation
    (Higham, "Accuracy and Stability of Numerical Algorithms", sec. 4.2) of
    the FP32 squares, padded with zeros to a power of two, computed here level
    by level over the whole array with numpy (the oracle walks tiles, lanes
    and a tile tree instead) -- any dropped element, wrong lane index or
    mis-paired add changes the bits;
  * its error against the exact float64 sum stays within the pairwise bound;
  * exact cases: integer squares whose every partial sum is exact; one
    nonzero element anywhere (ragged tails included);
  * the clip factor equals torch.nn.utils.clip_grad_norm_'s coefficient on
    gradients whose norm is an exact integer (read back from a unit entry);
  * the clipped step with a power-of-two factor equals the plain step on
    gradients pre-scaled exactly in BF16, for every recipe.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import HYPER


def bf16_of(x) -> np.ndarray:
    return O.bf16_round(np.asarray(x, np.float32))


def pairwise_f32(x: np.ndarray) -> np.float32:
    """Recursive pairwise summation of float32 values: pad with zeros to a
    power of two, then add adjacent pairs level by level in float32."""
    x = np.asarray(x, np.float32)
    if x.size == 0:
        return np.float32(0)
    p = 1 << int(math.ceil(math.log2(x.size)))
    y = np.zeros(p, np.float32)
    y[: x.size] = x
    while y.size > 1:
        y = (y[0::2] + y[1::2]).astype(np.float32)
    return y[0]


def squares(bits: np.ndarray) -> np.ndarray:
    g = (bits.astype(np.uint32) << 16).view(np.float32)
    return (g * g).astype(np.float32)


def textbook_sqnorm(grads) -> np.float32:
    total = np.float32(0)
    for b in grads:
        total = np.float32(total + pairwise_f32(squares(b)))
    return total


@pytest.mark.parametrize("sizes", [[1], [7], [256], [257], [1000, 3, 4096], [65536 + 129], [0, 5, 0, 300]])
def test_sqnorm_is_pairwise_summation(sizes):
    rng = np.random.default_rng(sum(sizes) + len(sizes))
    grads = [bf16_of(rng.standard_normal(n) * rng.choice([1e-3, 1.0, 30.0])) for n in sizes]
    got = O.grad_sqnorm(grads)
    want = textbook_sqnorm(grads)
    assert got.view(np.uint32) == want.view(np.uint32), (got, want)


def test_sqnorm_order_distinguishes_pairwise_from_sequential():
    # 4096^2 = 2^24 followed by 255 ones: sequential FP32 addition loses every
    # one (2^24 + 1 rounds to even), the pairwise tree keeps all but one:
    # lane 0 gives 2^24 + 6, the other 31 lanes 8 each, the lane tree adds
    # 8, 16, 32, 64, 128 to it.
    g = np.ones(256, np.float32)
    g[0] = 4096.0
    got = O.grad_sqnorm([bf16_of(g)])
    assert float(got) == 2.0 ** 24 + 254
    assert float(np.float32(np.cumsum(g.astype(np.float32) ** 2, dtype=np.float32)[-1])) == 2.0 ** 24


def test_sqnorm_error_bound_against_float64():
    rng = np.random.default_rng(5)
    sizes = [300000, 4097, 128, 1]
    grads = [bf16_of(rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 2)) for n in sizes]
    exact = sum(float(np.sum(squares(b).astype(np.float64))) for b in grads)
    got = float(O.grad_sqnorm(grads))
    # all terms >= 0: relative error <= (depth + tensors) u, depth = log2 of the
    # padded length, plus one rounding per square (exact here: 8-bit significands)
    depth = max(int(math.ceil(math.log2(n))) for n in sizes) + 8
    u = 2.0 ** -24
    assert abs(got - exact) <= (depth + len(sizes)) * u * exact
    assert got != 0


def test_sqnorm_exact_integer_cases():
    # squares of small integers: every partial sum is an integer below 2^24
    rng = np.random.default_rng(9)
    grads = [bf16_of(rng.integers(-20, 21, size=n).astype(np.float32)) for n in (1, 255, 256, 1031, 70000)]
    exact = sum(int(np.sum(squares(b).astype(np.int64))) for b in grads)
    assert exact < 2 ** 24
    assert float(O.grad_sqnorm(grads)) == exact


@pytest.mark.parametrize("n,pos", [(1, 0), (300, 299), (300, 255), (256 * 40 + 3, 256 * 40 + 2), (5000, 1234)])
def test_sqnorm_single_element(n, pos):
    g = np.zeros(n, np.float32)
    g[pos] = -3.5
    other = np.zeros(17, np.float32)
    assert float(O.grad_sqnorm([bf16_of(other), bf16_of(g), bf16_of(other)])) == 12.25


def test_sqnorm_empty_and_zero():
    assert float(O.grad_sqnorm([])) == 0.0
    assert float(O.grad_sqnorm([np.zeros(0, np.uint16)])) == 0.0
    assert float(O.grad_sqnorm([bf16_of(np.zeros(999))])) == 0.0


@pytest.mark.parametrize("triple,scale", [((1, 2, 2), 1.0), ((2, 3, 6), 0.25), ((1, 4, 8), 64.0), ((2, 6, 9), 2.0 ** -10)])
@pytest.mark.parametrize("max_norm", [1.0, 0.37, 5.0, 1e4])
def test_clip_factor_matches_torch(triple, scale, max_norm):
    a, b, c = triple
    vals = np.array([a, b, c], np.float64) * scale
    norm = math.sqrt(a * a + b * b + c * c) * scale        # an exact integer times a power of two
    sq = O.grad_sqnorm([bf16_of(vals)])
    assert float(sq) == norm * norm
    # torch: unit entry (scaled by `scale`) in its own parameter; its clipped
    # value divided by `scale` is the coefficient, exactly
    ps = [torch.nn.Parameter(torch.zeros(1)) for _ in range(3)]
    for p, x in zip(ps, vals):
        p.grad = torch.tensor([x], dtype=torch.float32)
    tn = torch.nn.utils.clip_grad_norm_(ps, max_norm)
    assert float(tn) == norm
    coef_torch = np.float32(float(ps[0].grad[0]) / vals[0])
    got = O.clip_factor(sq, max_norm)
    assert got.view(np.uint32) == coef_torch.view(np.uint32), (got, coef_torch)
    if max_norm >= norm + 1e-6:
        assert float(got) == 1.0


def test_clip_factor_special_values():
    assert float(O.clip_factor(0.0, 1.0)) == 1.0
    assert float(O.clip_factor(np.inf, 1.0)) == 0.0
    assert np.isnan(O.clip_factor(np.nan, 1.0))


@pytest.mark.parametrize("recipe,flags", [("zip_sr", 0), ("ze_eden", 0), ("torchao", 0), ("zip_sr", 1),
                                          ("factored", 0)])
def test_clipped_step_equals_prescaled_step(recipe, flags):
    """clip = 1/4 is exact on BF16 values (no subnormals here): stepping g with
    the clip factor must equal stepping the exactly pre-scaled g / 4."""
    rng = np.random.default_rng(17)
    rows, n = 3, 3 * 300
    fl = O.T_LM_HEAD | (O.T_FACTORED if recipe == "factored" else 0)
    p0 = rng.standard_normal(n).astype(np.float32)
    a = O.OracleTensor.zeros_state(p0, 7, rows=rows, flags=fl, recipe=recipe)
    b = O.OracleTensor.zeros_state(p0, 7, rows=rows, flags=fl, recipe=recipe)
    h = HYPER
    for t in (1, 2, 3):
        g = rng.standard_normal(n).astype(np.float32) * 0.01
        gb = bf16_of(g)
        gq = bf16_of((gb.astype(np.uint32) << 16).view(np.float32) * np.float32(0.25))
        a.step(gb, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 3, recipe, flags, clip=0.25)
        b.step(gq, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 3, recipe, flags)
        assert np.array_equal(a.param.view(np.uint32), b.param.view(np.uint32)), t
        assert np.array_equal(a.m_codes, b.m_codes) and np.array_equal(a.m_scale, b.m_scale)
        if a.factored:
            assert np.array_equal(a.v_row, b.v_row) and np.array_equal(a.v_col, b.v_col)
        else:
            assert np.array_equal(a.v_codes, b.v_codes) and np.array_equal(a.v_scale, b.v_scale)


def test_clip_one_is_the_plain_step():
    rng = np.random.default_rng(3)
    p0 = rng.standard_normal(500).astype(np.float32)
    a = O.OracleTensor.zeros_state(p0, 1)
    b = O.OracleTensor.zeros_state(p0, 1)
    h = HYPER
    for t in (1, 2):
        gb = bf16_of(rng.standard_normal(500) * 0.1)
        a.step(gb, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, "zip_sr", clip=1.0)
        b.step(gb, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, "zip_sr")
        assert np.array_equal(a.param.view(np.uint32), b.param.view(np.uint32))


def test_sqnorm_pairing_on_equal_magnitude_tiles():
    # with squares of one magnitude every pairing choice shows in the rounded
    # bits: 200 single-tile tensors (and ragged ones) against textbook pairwise
    rng = np.random.default_rng(77)
    for k in range(200):
        n = 256 if k % 4 else int(rng.integers(129, 256))
        g = bf16_of(rng.normal(0, 1, n))
        got = O.grad_sqnorm([g])
        want = textbook_sqnorm([g])
        assert got.view(np.uint32) == want.view(np.uint32), (k, got, want)


def test_sqnorm_lane_pairing_hand_derived():
    # BF16 squares carry at most 16 significant bits, so most lane sums are
    # exact whatever the pairing; this case makes the pairing visible.  Lane 0
    # holds 4096, 1, 2, 3 (squares 2^24, 1, 4, 9), everything else is 0.  The
    # stated order: (2^24 + 1) rounds to 2^24 (tie to even), 4 + 9 = 13, and
    # 2^24 + 13 rounds to 2^24 + 12 (tie to even).  Pairing (s0+s2), (s1+s3)
    # would give 2^24 + 14 exactly; left to right, 2^24 + 12 as well.
    g = np.zeros(256, np.float32)
    g[:4] = [4096.0, 1.0, 2.0, 3.0]
    assert float(O.grad_sqnorm([bf16_of(g)])) == 2.0 ** 24 + 12
