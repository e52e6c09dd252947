"""Parity of the CUDA step with the oracle at the full workload sizes.

Each workload is built exactly as bench.py builds it (one Q4State over the
whole tensor list, inputs drawn on the device by the seeded generators of
workloads.py, state zeroed) and stepped with the same single multi-tensor
launch bench.py times.  The oracle cannot run 8 billion parameters in a test,
so it checks samples it can compute on its own:

  * packed (ZIP-SR, ZE-EDEN, factored 1-D) tensors: blocks are independent,
    so for every tensor the first, the last and two seeded random blocks are
    stepped by the oracle as one-block tensors (elem_offset = the block's
    start, so the random draws are the same) from the same initial weights
    and gradients, and compared bit for bit after every one of 10 steps
    (the first, the second and the last of them included);
  * factored rank >= 2 tensors: their statistics span the whole tensor, so a
    subset of whole tensors (the embedding and every tensor of the first and
    last layer) is stepped by the oracle and compared with the factored
    tolerances of the small-list test.

Nothing the CUDA library writes is ever fed to the oracle: both sides start
from the generator's initial weights and read the generator's gradients, and
evolve on their own for all the steps.  The acceptance allows codes to differ
on elements within 1e-6 relative of a decision boundary; these tests allow no
such exception (every code, scale and weight bit-identical, factored weights
within 1e-6 max(1, |theta|)) and print the count of excepted elements, 0.
"""
import gc

import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import workloads as W
from oracle import oracle as O
from parity_util import HYPER, bf16_bits, bf16_close, neq_f32

pytestmark = pytest.mark.gpu

BLOCK = 128


def _build(w, dev):
    st = q4.Q4State(w.tensors, w.recipe, device=dev)
    for i, s in enumerate(w.tensors):
        st.view(i, "param").copy_(W.init_param(s, i, device=dev))
    st.init()
    return st


def _draw(w, st, t, dev):
    for i, s in enumerate(w.tensors):
        W.draw_grad(w, s, i, t, device=dev, out=st.view(i, "grad"))


def _sample_blocks(numel, rng):
    nb = (numel + BLOCK - 1) // BLOCK
    return sorted({0, nb - 1, *rng.integers(0, nb, size=2).tolist()})


def _free(st):
    del st
    gc.collect()
    torch.cuda.empty_cache()


def _run_packed(w, steps, flags, tensor_filter=None, max_grad_norm=None):
    """Step the whole workload on the GPU; check sampled blocks of the tensors
    tensor_filter accepts (all packed ones by default) against the oracle."""
    dev = torch.device("cuda", 0)
    st = _build(w, dev)
    rng = np.random.default_rng(1234)
    samples = []          # (tensor index, block, OracleTensor)
    for i, s in enumerate(w.tensors):
        factored = w.recipe == "factored" and bool(s.flags & W.T_FACTORED)
        if factored or (tensor_filter is not None and not tensor_filter(i, s)):
            continue
        th = st.view(i, "param")
        for b in _sample_blocks(s.numel, rng):
            lo, hi = b * BLOCK, min(b * BLOCK + BLOCK, s.numel)
            samples.append((i, b, O.OracleTensor.zeros_state(th[lo:hi].cpu().numpy(), i, rows=1, flags=s.flags,
                                                              elem_offset=lo, recipe=w.recipe)))
    h = HYPER
    checked = 0
    for t in range(w.first_step, w.first_step + steps):
        _draw(w, st, t, dev)
        grads = {}
        for i, b, _ in samples:
            if i not in grads:
                grads[i] = st.view(i, "grad")
        host_g = {}
        for i, b, o in samples:
            lo = b * BLOCK
            hi = lo + o.param.size
            host_g[(i, b)] = bf16_bits(grads[i][lo:hi])
        clip = None
        if max_grad_norm is not None:
            # the oracle's global sum of squares over every gradient of the workload
            sq = O.grad_sqnorm([bf16_bits(st.view(i, "grad")) for i in range(len(w.tensors))])
            clip = O.clip_factor(sq, max_grad_norm)
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=0, flags=flags,
                max_grad_norm=max_grad_norm)
        torch.cuda.synchronize()
        assert st.status() == 0
        if max_grad_norm is not None:
            got = np.float32(st.sqnorm.cpu().numpy()[0])
            assert got.view(np.uint32) == sq.view(np.uint32), (w.name, t, got, sq)
            assert float(clip) < 1.0
        for i, b, o in samples:
            o.step(host_g[(i, b)], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, w.recipe,
                   flags, clip=clip)
            lo, n = b * BLOCK, o.param.size
            th = st.view(i, "param")[lo:lo + n].cpu().numpy()
            assert not neq_f32(th, o.param).any(), (w.name, i, b, t, "param")
            assert np.array_equal(bf16_bits(st.view(i, "param_bf16")[lo:lo + n]), o.param_bf16), (w.name, i, b, t)
            mc = st.view(i, "m_codes")[b * 64:(b + 1) * 64].cpu().numpy()
            assert np.array_equal(mc, o.m_codes), (w.name, i, b, t, "m_codes")
            ms = st.view(i, "m_scale")[b:b + 1].cpu().numpy()
            assert not neq_f32(ms, o.m_scale).any(), (w.name, i, b, t, "m_scale")
            vc = st.view(i, "v_codes")[b * 64:(b + 1) * 64].cpu().numpy()
            assert np.array_equal(vc, o.v_codes), (w.name, i, b, t, "v_codes")
            vs = st.view(i, "v_scale")[b:b + 1].cpu().numpy()
            assert not neq_f32(vs, o.v_scale).any(), (w.name, i, b, t, "v_scale")
            checked += 1
    _free(st)
    print(f"{w.name}: {steps} steps, {checked} block comparisons, {checked * BLOCK} element comparisons per "
          f"quantity, excepted elements: 0")
    return checked


STEPS = 10


def test_gpt1p4b_zipsr_lm_head_sr_sampled_blocks():
    w = W.WORKLOADS["gpt1p4b_zipsr"]
    n = _run_packed(w, STEPS, q4.Q4_LM_HEAD_SR_ACTIVE)
    assert n >= STEPS * 4 * 100


def test_gpt1p4b_zipsr_clipped_sampled_blocks():
    # global-norm clipping at the full 1.4B size: the GPU's sum of squares over
    # all 1.4B gradients equals the oracle's bit for bit, and sampled blocks of
    # the clipped step match
    w = W.WORKLOADS["gpt1p4b_zipsr"]
    n = _run_packed(w, 3, q4.Q4_LM_HEAD_SR_ACTIVE, max_grad_norm=1e-3)
    assert n >= 3 * 4 * 100


def test_gpt1p4b_torchao_sampled_blocks():
    # the TorchAO baseline recipe at the full 1.4B size (LM head flagged, final
    # phase active: it stays RTN in this recipe)
    w = W.WORKLOADS["gpt1p4b_torchao"]
    n = _run_packed(w, STEPS, q4.Q4_LM_HEAD_SR_ACTIVE)
    assert n >= STEPS * 4 * 100


@pytest.mark.parametrize("variant", ["m_sr_all", "v_update_rtn", "v_next_r", "v_next_r_update_rtn"])
def test_gpt1p4b_rounding_variants_sampled_blocks(variant):
    # the rounding variants at the full 1.4B size, on the same launch path as
    # bench.py --variant (their full tiles take the fast path)
    fl = {"m_sr_all": q4.Q4_M_SR_ALL, "v_update_rtn": q4.Q4_V_UPDATE_RTN, "v_next_r": q4.Q4_V_NEXT_R,
          "v_next_r_update_rtn": q4.Q4_V_NEXT_R | q4.Q4_V_UPDATE_RTN}[variant]
    w = W.WORKLOADS["gpt1p4b_zipsr"]
    n = _run_packed(w, 3, q4.Q4_LM_HEAD_SR_ACTIVE | fl)
    assert n >= 3 * 4 * 100


@pytest.mark.parametrize("name", ["llama8b_zipsr", "llama8b_zeeden"])
def test_llama8b_sampled_blocks(name):
    w = W.WORKLOADS[name]
    n = _run_packed(w, STEPS, 0)
    assert n >= STEPS * 4 * 100


def test_qwen0p6b_factored_whole_tensors_and_sampled_blocks():
    w = W.WORKLOADS["qwen0p6b_factored"]
    dev = torch.device("cuda", 0)
    st = _build(w, dev)
    per_layer = 11
    last0 = 1 + 27 * per_layer
    whole = [0, *range(1, 1 + per_layer), *range(last0, last0 + per_layer), len(w.tensors) - 1]
    ora = {}
    for i in whole:
        s = w.tensors[i]
        ora[i] = O.OracleTensor.zeros_state(st.view(i, "param").cpu().numpy(), i, rows=s.rows, flags=s.flags,
                                            recipe="factored")
    rng = np.random.default_rng(99)
    blocks = []
    for i, s in enumerate(w.tensors):
        if i in ora or (s.flags & W.T_FACTORED):
            continue
        th = st.view(i, "param")
        for b in _sample_blocks(s.numel, rng):
            lo, hi = b * BLOCK, min(b * BLOCK + BLOCK, s.numel)
            blocks.append((i, b, O.OracleTensor.zeros_state(th[lo:hi].cpu().numpy(), i, rows=1, flags=s.flags,
                                                             elem_offset=lo, recipe="factored")))
    h = HYPER
    worst = 0.0
    for t in range(1, STEPS + 1):
        _draw(w, st, t, dev)
        host_g = {i: bf16_bits(st.view(i, "grad")) for i in ora}
        host_b = {(i, b): bf16_bits(st.view(i, "grad")[b * BLOCK:b * BLOCK + o.param.size]) for i, b, o in blocks}
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=0)
        torch.cuda.synchronize()
        assert st.status() == 0
        for i, o in ora.items():
            o.step(host_g[i], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, "factored")
            assert np.array_equal(st.view(i, "m_codes").cpu().numpy(), o.m_codes), (i, t)
            assert not neq_f32(st.view(i, "m_scale").cpu().numpy(), o.m_scale).any(), (i, t)
            th = st.view(i, "param").cpu().numpy()
            d = np.abs(th.astype(np.float64) - o.param)
            assert (d <= 1e-6 * np.maximum(1.0, np.abs(o.param))).all(), (i, t, float(d.max()))
            worst = max(worst, float(d.max(initial=0.0)))
            assert bf16_close(bf16_bits(st.view(i, "param_bf16")), o.param_bf16).all(), (i, t)
            if o.factored:
                R = st.view(i, "v_row").cpu().numpy().astype(np.float64)
                C = st.view(i, "v_col").cpu().numpy().astype(np.float64)
                assert (np.abs(R - o.v_row) <= 1e-5 * np.abs(o.v_row)).all(), (i, t)
                assert (np.abs(C - o.v_col) <= 1e-5 * np.abs(o.v_col)).all(), (i, t)
            else:
                assert np.array_equal(st.view(i, "v_codes").cpu().numpy(), o.v_codes), (i, t)
                assert not neq_f32(st.view(i, "v_scale").cpu().numpy(), o.v_scale).any(), (i, t)
        for i, b, o in blocks:
            o.step(host_b[(i, b)], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, "factored")
            lo, n = b * BLOCK, o.param.size
            assert not neq_f32(st.view(i, "param")[lo:lo + n].cpu().numpy(), o.param).any(), (i, b, t)
            assert np.array_equal(st.view(i, "v_codes")[b * 64:(b + 1) * 64].cpu().numpy(), o.v_codes), (i, b, t)
    _free(st)
    n_whole = sum(w.tensors[i].numel for i in ora)
    print(f"qwen0p6b_factored: {STEPS} steps, {len(ora)} whole tensors ({n_whole} elements, max |dtheta| "
          f"{worst:.3g}) and {len(blocks)} sampled 1-D blocks, excepted elements: 0")


def test_mat4096_zeeden_full_size_hundred_steps():
    # the 4096 x 4096 ZE-EDEN matrix (16.8M parameters, row-scaled gradients,
    # 5% zero blocks) at its full size for all 100 steps; both sides run
    # free, compared element by element at steps 1, 2, 3, 10, 50 and 100
    from parity_util import Pair, grads_for
    w = W.WORKLOADS["mat4096_zeeden"]
    p = Pair(w.tensors, w.recipe)
    checked = []
    for t in range(1, 101):
        p.step(t, grads_for(w, t))
        if t in (1, 2, 3, 10, 50, 100):
            r = p.compare()
            assert r["codes"] == 0 and r["scales"] == 0 and r["theta"] == 0 and r["bf16"] == 0, (t, r)
            checked.append(t)
    print(f"mat4096_zeeden: 100 steps, {w.tensors[0].numel} elements compared at steps {checked}, "
          f"excepted elements: 0")


def test_tensor_beyond_2_pow_31_elements_sampled_blocks():
    # one 1-D tensor of 2^31 + 2^20 + 37 elements (64-bit element offsets in
    # the tile list, the copy sources and the Philox counters; a ragged last
    # block), flagged as the LM head with its SR phase active, so both draw
    # purposes run at element indices above 2^31.  Blocks on both sides of
    # element 2^31, the first and the last block are stepped by the oracle for
    # 3 steps and compared bit for bit.
    n = 2 ** 31 + 2 ** 20 + 37
    w = W.custom("big", [(n,)], "zip_sr", flags=[W.T_LM_HEAD])
    dev = torch.device("cuda", 0)
    st = _build(w, dev)
    nb = (n + BLOCK - 1) // BLOCK
    edge = 2 ** 31 // BLOCK
    blocks = [0, edge - 1, edge, edge + 1, nb - 1]
    th = st.view(0, "param")
    ora = {b: O.OracleTensor.zeros_state(th[b * BLOCK:min(b * BLOCK + BLOCK, n)].cpu().numpy(), 0, rows=1,
                                         flags=W.T_LM_HEAD, elem_offset=b * BLOCK, recipe="zip_sr")
           for b in blocks}
    h = HYPER
    for t in range(1, 4):
        _draw(w, st, t, dev)
        g = st.view(0, "grad")
        host_g = {b: bf16_bits(g[b * BLOCK:b * BLOCK + o.param.size]) for b, o in ora.items()}
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=0,
                flags=q4.Q4_LM_HEAD_SR_ACTIVE)
        torch.cuda.synchronize()
        assert st.status() == 0
        for b, o in ora.items():
            o.step(host_g[b], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 0, "zip_sr",
                   q4.Q4_LM_HEAD_SR_ACTIVE)
            lo, k = b * BLOCK, o.param.size
            assert not neq_f32(st.view(0, "param")[lo:lo + k].cpu().numpy(), o.param).any(), (b, t)
            assert np.array_equal(bf16_bits(st.view(0, "param_bf16")[lo:lo + k]), o.param_bf16), (b, t)
            assert np.array_equal(st.view(0, "m_codes")[b * 64:(b + 1) * 64].cpu().numpy(), o.m_codes), (b, t)
            assert np.array_equal(st.view(0, "v_codes")[b * 64:(b + 1) * 64].cpu().numpy(), o.v_codes), (b, t)
            assert not neq_f32(st.view(0, "m_scale")[b:b + 1].cpu().numpy(), o.m_scale).any(), (b, t)
            assert not neq_f32(st.view(0, "v_scale")[b:b + 1].cpu().numpy(), o.v_scale).any(), (b, t)
    _free(st)
    print(f"big tensor of {n} elements: 3 steps, {len(blocks)} blocks per step bit-identical, excepted elements: 0")


def test_factored_tensor_beyond_2_pow_31_elements_closed_form():
    # a factored [65537, 32768] parameter (2^31 + 32768 elements: 64-bit matrix
    # positions in the statistics pass, 257 column slabs, mean(R) over 65537
    # rows, the step's (row, column) tracking past element 2^31) with every
    # gradient 2^-4 (exact in BF16).  Closed forms after one step from zero
    # state: every row and column mean of g^2 is 2^-8 exactly, so every R_i
    # and C_j is omb2 * 2^-8 exactly; every m' is omb1 * 2^-4, so every NF4
    # code is 15 and every m scale m'; theta follows AdamW with vhat = R_i C_j
    # / mean(R) = omb2 * 2^-8 (up to the rounding of mean(R)), checked within
    # the factored tolerance on blocks around element 2^31 and at both ends.
    rows, cols = 65537, 32768
    n = rows * cols
    w = W.custom("bigf", [(rows, cols)], "factored", flags=[W.T_FACTORED])
    dev = torch.device("cuda", 0)
    st = _build(w, dev)
    g = 2.0 ** -4
    st.view(0, "grad").fill_(g)
    nb = n // BLOCK
    edge = 2 ** 31 // BLOCK
    blocks = [0, edge - 1, edge, edge + 1, nb - 1]
    th0 = {b: st.view(0, "param")[b * BLOCK:(b + 1) * BLOCK].cpu().numpy().astype(np.float64) for b in blocks}
    h = HYPER
    st.step(1, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=0)
    torch.cuda.synchronize()
    assert st.status() == 0
    # the host scalars as the library forms them: from the FP32 arguments, in
    # double, each rounded once to FP32
    f32 = np.float32
    lr, b1, b2, eps, wd = (float(f32(h[k])) for k in ("lr", "beta1", "beta2", "eps", "weight_decay"))
    omb1, omb2 = f32(1.0 - b1), f32(1.0 - b2)
    x = f32(omb2 * f32(2.0 ** -8))
    R = st.view(0, "v_row").cpu().numpy()
    C = st.view(0, "v_col").cpu().numpy()
    assert R.shape == (rows,) and C.shape == (cols,)
    assert (R == x).all() and (C == x).all(), (R.min(), R.max(), C.min(), C.max(), x)
    m1 = f32(omb1 * f32(g))
    c2 = f32(1.0 / np.sqrt(1.0 - b2))
    step_size = f32(lr / (1.0 - b1))
    decay = f32(1.0 - lr * wd)
    r = 1.0 / (np.sqrt(float(x)) * float(c2) + eps)
    for b in blocks:
        th = st.view(0, "param")[b * BLOCK:(b + 1) * BLOCK].cpu().numpy().astype(np.float64)
        want = th0[b] * float(decay) - float(step_size) * float(m1) * r
        assert (np.abs(th - want) <= 1e-6 * np.maximum(1.0, np.abs(want))).all(), (b, np.abs(th - want).max())
        assert (st.view(0, "m_codes")[b * 64:(b + 1) * 64].cpu().numpy() == 0xFF).all(), b
        assert st.view(0, "m_scale")[b:b + 1].cpu().numpy()[0] == m1, b
    _free(st)
    print(f"factored tensor of {n} elements: R, C exact on all {rows} rows and {cols} columns; "
          f"{len(blocks)} blocks within the factored tolerance")
