"""Pins of the oracle's factored second moment, through its C step.

AReno docs "4-bit AdamW", section "State representation": a rank >= 2
parameter keeps Adafactor-style statistics instead of a packed v -- the row
means R and column means C of g^2 over the [shape[0], -1] view, each an
exponential average -- and the update uses vhat_ij = R_i * C_j / mean_i(R_i);
1-D parameters keep a packed 4-bit v in a map that excludes zero.

Every expectation below is restated here in numpy from those definitions and
compared with the weights (and codes) the oracle's C step writes:
  * the weights after steps 1..3 on a square tensor with unequal row and
    column scales (a swapped row/column index or a product in place of the
    quotient changes vhat by large factors), and on a wide one;
  * mean(R) = 0 gives vhat = 0 (beta2 = 0 makes R the current step's means,
    so a zero gradient after a nonzero one reaches mean(R) = 0 with m != 0);
  * a 1-D tensor under the factored recipe stores the nearest zero-excluding
    Dyn4-NZ level, never the zero-inclusive Dyn4 one, and its next step
    decodes that level.
The square-tensor test comes first: a planted row/column swap fails there
before a non-square shape could read past R.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O

H = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _from_bf16(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _decode(packed, scales, levels, n):
    e = np.arange(n)
    q = (packed[e >> 1] >> (4 * (e & 1))) & 15
    return (levels[q].astype(np.float32) * scales[e // 128].astype(np.float32)).astype(np.float32)


def _codes(packed, n):
    e = np.arange(n)
    return (packed[e >> 1] >> (4 * (e & 1))) & 15


def _scalars(t, beta1, beta2, lr=H["lr"], wd=H["wd"]):
    d1, d2 = float(np.float32(beta1)), float(np.float32(beta2))
    lr, wd = float(np.float32(lr)), float(np.float32(wd))
    return dict(c2=1.0 / np.sqrt(1.0 - d2 ** t), step_size=lr / (1.0 - d1 ** t), decay=1.0 - lr * wd,
                b1=d1, b2=d2)


def _factored_run(rows, cols, grads, beta2=H["beta2"], steps=None):
    """Steps the oracle on one factored [rows, cols] tensor and checks theta
    after every step against a float64 restatement of AdamW with
    vhat_ij = R_i C_j / mean(R), R and C the exponential averages of the row
    and column means of g^2.  The first moment is the oracle's decoded state
    (m is quantised between steps)."""
    rng = np.random.default_rng(11)
    n = rows * cols
    t = O.OracleTensor.zeros_state(rng.normal(0, 0.02, n).astype(np.float32), 3, rows=rows, flags=O.T_FACTORED,
                                   recipe="factored")
    assert t.factored and t.v_codes is None
    nf4 = O.codebooks()["nf4"]
    R = np.zeros(rows)
    C = np.zeros(cols)
    worst = 0.0
    for k, g in enumerate(grads):
        step = k + 1
        m_dec = _decode(t.m_codes, t.m_scale, nf4, n).astype(np.float64)
        theta = t.param.astype(np.float64)
        t.step(g, H["lr"], H["beta1"], beta2, H["eps"], H["wd"], step, 0, "factored")
        s = _scalars(step, H["beta1"], beta2)
        gf = _from_bf16(g).astype(np.float64).reshape(rows, cols)
        R = s["b2"] * R + (1 - s["b2"]) * (gf ** 2).mean(axis=1)
        C = s["b2"] * C + (1 - s["b2"]) * (gf ** 2).mean(axis=0)
        rbar = R.mean()
        vhat = np.zeros((rows, cols)) if rbar == 0 else R[:, None] * C[None, :] / rbar
        m1 = s["b1"] * m_dec + (1 - s["b1"]) * gf.reshape(-1)
        r = 1.0 / (np.sqrt(vhat.reshape(-1)) * s["c2"] + H["eps"])
        want = theta * s["decay"] - s["step_size"] * m1 * r
        d = np.abs(t.param.astype(np.float64) - want)
        worst = max(worst, float((d / np.maximum(1.0, np.abs(want))).max()))
        assert np.all(d <= 1e-6 * np.maximum(1.0, np.abs(want))), (step, float(d.max()))
        # the statistics themselves (float64 restatement, FP32 storage)
        assert np.allclose(t.v_row, R, rtol=1e-5, atol=0) and np.allclose(t.v_col, C, rtol=1e-5, atol=0), step
    return t, worst


def test_factored_square_tensor_matches_float64_restatement():
    # unequal row and column scales over two decades each, so that R_i C_j
    # and R_j C_i differ and vhat is far from mean(R)
    rows = cols = 48
    rng = np.random.default_rng(12)
    sig_r = 10.0 ** rng.uniform(-1, 1, rows)
    sig_c = 10.0 ** rng.uniform(-1, 1, cols)
    grads = [_bf16((rng.normal(0, 1e-3, (rows, cols)) * sig_r[:, None] * sig_c[None, :]).reshape(-1))
             for _ in range(3)]
    t, _ = _factored_run(rows, cols, grads)
    # the test has teeth: the swapped-index and product-for-quotient forms are
    # far outside the tolerance on this input
    R, C = t.v_row.astype(np.float64), t.v_col.astype(np.float64)
    rbar = R.mean()
    right = R[:, None] * C[None, :] / rbar
    swapped = R[None, :] * C[:, None] / rbar
    assert np.max(np.abs(np.sqrt(swapped) - np.sqrt(right)) / np.sqrt(right)) > 1.0
    assert rbar < 1e-6   # product and quotient by mean(R) differ by a factor above 1e12


@pytest.mark.parametrize("rows,cols", [(24, 200), (130, 64), (1, 384)])
def test_factored_rectangular_tensor_matches_float64_restatement(rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    sig_r = 10.0 ** rng.uniform(-1, 1, rows)
    sig_c = 10.0 ** rng.uniform(-1, 1, cols)
    grads = [_bf16((rng.normal(0, 1e-3, (rows, cols)) * sig_r[:, None] * sig_c[None, :]).reshape(-1))
             for _ in range(3)]
    _factored_run(rows, cols, grads)


def test_factored_rank1_gradient_gives_exact_vhat_on_the_first_step():
    # g_ij = a_i b_j (exact in BF16): after step 1 vhat = (1 - beta2) g_ij^2,
    # so the update is the unquantised first AdamW step: theta' = theta decay
    # - step (1-b1) g / (sqrt((1-b2) g^2) c2 + eps)
    rows, cols = 16, 32
    a = 2.0 ** np.arange(-4, 12, dtype=np.float64)[:rows] * 2.0 ** -13
    b = 2.0 ** (np.arange(cols) % 5 - 2.0)
    g = _bf16((a[:, None] * b[None, :]).reshape(-1))
    assert np.array_equal(_from_bf16(g).astype(np.float64), (a[:, None] * b[None, :]).reshape(-1))
    _factored_run(rows, cols, [g])


def test_zero_mean_of_r_gives_zero_vhat():
    # beta2 = 0: R and C are this step's means.  Step 1 with a nonzero
    # gradient leaves m != 0; step 2 with g = 0 gives R = C = 0, mean(R) = 0,
    # vhat = 0 by definition, so r = 1 / eps and theta' = theta decay -
    # step (m' (1/eps)), m' = beta1 m.  Restated in FP32 operation by
    # operation (numpy float32), so the weights must agree bit for bit.
    rows, cols = 8, 256
    n = rows * cols
    rng = np.random.default_rng(13)
    t = O.OracleTensor.zeros_state(rng.normal(0, 0.02, n).astype(np.float32), 1, rows=rows, flags=O.T_FACTORED,
                                   recipe="factored")
    g1 = _bf16(rng.normal(0, 1e-3, n))
    t.step(g1, H["lr"], H["beta1"], 0.0, H["eps"], H["wd"], 1, 0, "factored")
    m_dec = _decode(t.m_codes, t.m_scale, O.codebooks()["nf4"], n)
    assert np.count_nonzero(m_dec) > n // 2
    theta = t.param.copy()
    t.step(np.zeros(n, np.uint16), H["lr"], H["beta1"], 0.0, H["eps"], H["wd"], 2, 0, "factored")
    assert np.all(t.v_row == 0) and np.all(t.v_col == 0)
    h = O.host_scalars(H["lr"], H["beta1"], 0.0, H["wd"], 2)
    f = np.float32
    m1 = (f(H["beta1"]) * m_dec).astype(np.float32)            # fma(b1, m, (1-b1) 0) = RN(b1 m)
    r = f(1.0) / (f(0.0) * f(h["c2"]) + f(H["eps"]))
    want = (theta * f(h["decay"])).astype(np.float32) - (f(h["step_size"]) * (m1 * r).astype(np.float32))
    assert np.array_equal(t.param.view(np.uint32), want.astype(np.float32).view(np.uint32))
    # the update is large (r = 1e8): a vhat of 1 in place of 0 would not be
    moved = np.abs(t.param.astype(np.float64) - (theta * f(h["decay"])).astype(np.float64))
    assert moved.max() > 1e-2


def test_all_zero_gradients_only_decay_the_weights():
    rows, cols = 4, 128
    n = rows * cols
    rng = np.random.default_rng(14)
    th0 = rng.normal(0, 0.02, n).astype(np.float32)
    t = O.OracleTensor.zeros_state(th0, 2, rows=rows, flags=O.T_FACTORED, recipe="factored")
    for step in (1, 2):
        before = t.param.copy()
        t.step(np.zeros(n, np.uint16), H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], step, 0, "factored")
        h = O.host_scalars(H["lr"], H["beta1"], H["beta2"], H["wd"], step)
        assert np.array_equal(t.param, (before * np.float32(h["decay"])).astype(np.float32))
        assert np.all(t.m_scale == 0) and np.all(t.v_row == 0) and np.all(t.v_col == 0)


def _band_gradient(n, rng):
    """BF16 gradients whose v' = (1-b2) g^2 puts, in every block, elements in
    the band (0.0005, 0.00055) * max v' where the nearest Dyn4-NZ level (1e-4,
    code 0) and the nearest Dyn4 level (0.001, code 1; Dyn4's code 0 is 0)
    differ, plus elements below 0.0005 * max (Dyn4: level 0)."""
    g = rng.normal(0, 1e-3, n)
    for b in range(0, n, 128):
        g[b] = 1e-2                                                    # the block maximum
        g[b + 1:b + 9] = 1e-2 * np.sqrt(rng.uniform(0.000505, 0.000545, 8))   # inside the band
        g[b + 9:b + 13] = 1e-2 * np.sqrt(rng.uniform(0.00001, 0.0004, 4))     # below it
        g[b + 13:b + 128] = np.clip(np.abs(g[b + 13:b + 128]), 0, 9e-3) * np.sign(g[b + 13:b + 128])
    return _bf16(g)


def test_factored_1d_tensor_stores_nearest_zero_excluding_level():
    # AReno docs "State representation": 1-D tensors keep packed v in the
    # zero-excluding map (Dyn4-NZ) with RTN.  After step 1 from zero,
    # v' = (1-b2) g^2: each stored code is the nearest Dyn4-NZ level of v' at
    # the block scale max v'; step 2 decodes that level (never 0).
    n = 128 * 6 + 40
    rng = np.random.default_rng(15)
    g1 = _band_gradient(n, rng)
    t = O.OracleTensor.zeros_state(rng.normal(0, 0.02, n).astype(np.float32), 4, rows=1, flags=0,
                                   recipe="factored")
    assert not t.factored and t.v_codes is not None
    t.step(g1, H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], 1, 0, "factored")
    cb = O.codebooks()
    L = cb["dyn4nz"].astype(np.float64)
    assert L.min() > 0
    gf = _from_bf16(g1).astype(np.float64)
    v1 = float(np.float32(1.0 - float(np.float32(H["beta2"])))) * gf * gf
    q = _codes(t.v_codes, n)
    in_band = 0
    for b in range(O.nblocks(n)):
        sl = slice(128 * b, min(128 * b + 128, n))
        s = v1[sl].max()
        assert abs(t.v_scale[b] - s) <= 1e-6 * s           # no EDEN factor on factored 1-D v
        d = np.abs(v1[sl][:, None] - L[None, :] * s)
        assert np.all(d[np.arange(q[sl].size), q[sl]] <= d.min(1) + 1e-6 * s)
        y = v1[sl] / s
        in_band += int(((y > 0.0005 * (1 + 1e-4)) & (y < 0.00055 * (1 - 1e-4))).sum())
    assert in_band >= 8 * 6
    # step 2: v decodes as Dyn4-NZ level * scale
    v_dec = _decode(t.v_codes, t.v_scale, cb["dyn4nz"], n).astype(np.float64)
    assert np.all(v_dec > 0)
    m_dec = _decode(t.m_codes, t.m_scale, cb["nf4"], n).astype(np.float64)
    theta = t.param.astype(np.float64)
    g2 = _band_gradient(n, rng)
    t.step(g2, H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], 2, 0, "factored")
    s = _scalars(2, H["beta1"], H["beta2"])
    gf2 = _from_bf16(g2).astype(np.float64)
    m1 = s["b1"] * m_dec + (1 - s["b1"]) * gf2
    v2 = s["b2"] * v_dec + (1 - s["b2"]) * gf2 * gf2
    want = theta * s["decay"] - s["step_size"] * m1 / (np.sqrt(v2) * s["c2"] + H["eps"])
    assert np.all(np.abs(t.param - want) <= 1e-6 * np.maximum(1.0, np.abs(want)))


# ------------------------------------------------- data-parallel shards
# AReno docs "State representation": under data parallelism each rank's row
# and column sums of g^2 are added over the group, and R and C are updated
# from the totals.  A shard is a block-aligned run of the flattened parameter (it may
# start and end inside a row); every rank keeps the whole R and C.

def _exact_grad(n, rng, scale=2.0 ** -12):
    # small integers times a power of two: the squares and every sum of them
    # are exact in float64, so the order of the additions cannot matter
    return _bf16(rng.integers(-200, 201, n).astype(np.float64) * scale)


def test_shard_partials_equal_brute_force_sums():
    rows, cols = 40, 200
    n = rows * cols
    rng = np.random.default_rng(16)
    g = _bf16(rng.normal(0, 1e-3, n))
    gf = _from_bf16(g).astype(np.float64)
    for lo, hi in ((0, 128 * 7), (128 * 7, 128 * 33), (128 * 33, n)):
        t = O.OracleTensor.zeros_state(np.zeros(hi - lo, np.float32), 0, rows=rows, flags=O.T_FACTORED,
                                       elem_offset=lo, recipe="factored", cols=cols)
        rs, cs = t.factored_partials(g[lo:hi])
        e = np.arange(lo, hi)
        want_r = np.bincount(e // cols, weights=gf[lo:hi] ** 2, minlength=rows)
        want_c = np.bincount(e % cols, weights=gf[lo:hi] ** 2, minlength=cols)
        assert np.allclose(rs, want_r, rtol=1e-14, atol=0) and np.allclose(cs, want_c, rtol=1e-14, atol=0)
        assert np.all(rs[: lo // cols] == 0) and np.all(rs[(hi - 1) // cols + 1:] == 0)


@pytest.mark.parametrize("flags,call_flags", [(O.T_FACTORED, 0), (O.T_FACTORED | O.T_LM_HEAD, O.LM_HEAD_SR_ACTIVE)])
def test_sharded_factored_steps_equal_the_whole_tensor(flags, call_flags):
    # three shards cut inside rows (cols = 200); each step: every shard's
    # partial sums are added up, then each shard steps from the sums.  With
    # exact sums the shards reproduce the whole-tensor step bit for bit.
    rows, cols = 48, 200
    n = rows * cols
    cuts = [0, 128 * 23, 128 * 50, n]
    rng = np.random.default_rng(17)
    th0 = rng.normal(0, 0.02, n).astype(np.float32)
    whole = O.OracleTensor.zeros_state(th0, 7, rows=rows, flags=flags, recipe="factored")
    shards = [O.OracleTensor.zeros_state(th0[a:b], 7, rows=rows, flags=flags, elem_offset=a, recipe="factored",
                                         cols=cols) for a, b in zip(cuts, cuts[1:])]
    for step in range(1, 4):
        g = _exact_grad(n, rng)
        whole.step(g, H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], step, 3, "factored", call_flags)
        rs = np.zeros(rows)
        cs = np.zeros(cols)
        for sh, a, b in zip(shards, cuts, cuts[1:]):
            r, c = sh.factored_partials(g[a:b])
            rs += r
            cs += c
        for sh, a, b in zip(shards, cuts, cuts[1:]):
            sh.step_sums(g[a:b], rs, cs, H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], step, 3, "factored",
                         call_flags)
            assert np.array_equal(sh.param.view(np.uint32), whole.param[a:b].view(np.uint32)), (step, a)
            assert np.array_equal(sh.param_bf16, whole.param_bf16[a:b]), (step, a)
            assert np.array_equal(sh.m_codes, whole.m_codes[a // 2:b // 2 + (b - a) % 2]), (step, a)
            assert np.array_equal(sh.m_scale, whole.m_scale[a // 128:(b + 127) // 128]), (step, a)
            assert np.array_equal(sh.v_row, whole.v_row) and np.array_equal(sh.v_col, whole.v_col), (step, a)


def test_shard_step_of_a_packed_tensor_is_the_plain_step():
    n = 128 * 9
    rng = np.random.default_rng(18)
    th0 = rng.normal(0, 0.02, n).astype(np.float32)
    a = O.OracleTensor.zeros_state(th0, 2, elem_offset=256, recipe="factored")
    b = O.OracleTensor.zeros_state(th0, 2, elem_offset=256, recipe="factored")
    for step in (1, 2):
        g = _bf16(rng.normal(0, 1e-3, n))
        a.step(g, H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], step, 0, "factored")
        b.step_sums(g, np.zeros(1), np.zeros(1), H["lr"], H["beta1"], H["beta2"], H["eps"], H["wd"], step, 0,
                    "factored")
        assert np.array_equal(a.param, b.param) and np.array_equal(a.v_codes, b.v_codes)
