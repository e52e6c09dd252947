"""GPU-versus-oracle parity of the fused step through the C ABI.

Codes, scales, FP32 weights and BF16 weights must be bit-identical to the
oracle (both sides evaluate the same FP32 operation sequence; decisions that
turn floating point into codes are taken in FP32 on both).  The factored
statistics R, C are FP32 tree sums on the GPU and float64 sums in the oracle:
they are compared at 1e-5 relative, and the weights of factored tensors at
the stated bound |dtheta| <= 1e-6 * max(1, |theta|).
"""
import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import workloads as W
from parity_util import HYPER, Pair, grads_for

pytestmark = pytest.mark.gpu


def _assert_exact(res, step):
    assert res["codes"] == 0, (step, res)
    assert res["scales"] == 0, (step, res)
    assert res["theta"] == 0, (step, res)
    assert res["bf16"] == 0, (step, res)


def test_vec4096_zipsr_ten_steps_bit_exact():
    w = W.WORKLOADS["vec4096_zipsr"]
    p = Pair(w.tensors, w.recipe)
    for t in range(1, 11):
        p.step(t, grads_for(w, t), seed=0)
        _assert_exact(p.compare(), t)


def test_mat_zeeden_hundred_steps_bit_exact():
    # 1024 x 4096 slice of the 4096 x 4096 ZE-EDEN workload (same recipe, row
    # scales and 5% zero blocks), all 100 steps compared element by element.
    base = W.WORKLOADS["mat4096_zeeden"]
    w = W.custom("mat1024", [(1024, 4096)], "ze_eden", grad="row_scaled", sigma=(1e-6, 1e-2),
                 zero_block_frac=0.05)
    assert w.recipe == base.recipe
    p = Pair(w.tensors, w.recipe)
    for t in range(1, 101):
        p.step(t, grads_for(w, t))
        if t <= 5 or t % 10 == 0:
            _assert_exact(p.compare(), t)


RAGGED = [(1,), (5,), (127,), (128,), (129,), (255,), (256,), (1000,), (3, 129), (257, 7), (4096 + 64,),
          (7, 128), (128 * 13 + 17,)]


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "torchao"])
@pytest.mark.parametrize("sr", [False, True])
def test_ragged_tensor_list(recipe, sr):
    flags = [W.T_LM_HEAD if i % 3 == 0 else 0 for i in range(len(RAGGED))]
    w = W.custom("rag", RAGGED, recipe, flags=flags, grad="normal", sigma=(1e-3, 1e-3))
    offs = [128 * 5 * i for i in range(len(RAGGED))]
    p = Pair(w.tensors, recipe, elem_offsets=offs, tensor_ids=[10 + i for i in range(len(RAGGED))])
    for t in range(1, 8):
        p.step(t, grads_for(w, t, tids=[10 + i for i in range(len(RAGGED))]), seed=77,
               flags=1 if sr else 0)
        _assert_exact(p.compare(), t)


def test_lm_head_sr_phase_gpt_like():
    # LM-head SR active from the start of the final phase (steps 9001..), as in
    # the GPT-style 1.4B workload, on a reduced tensor list.
    shapes = [(512, 256), (256,), (768, 256), (256,)]
    flags = [W.T_LM_HEAD, 0, 0, 0]
    w = W.custom("gptmini", shapes, "zip_sr", flags=flags, grad="tensor_scaled", sigma=(1e-5, 1e-2))
    p = Pair(w.tensors, "zip_sr")
    for t in range(9001, 9006):
        p.step(t, grads_for(w, t), seed=3, flags=1)
        _assert_exact(p.compare(), t)


def test_degenerate_values():
    # zero, tiny (slow-path scales), huge, overflowing and mixed-magnitude
    # gradients.  Blocks 6 and 7 hold gradients whose square overflows FP32:
    # v' = +inf there, r = 0, a +inf (ZE-EDEN: NaN) v scale, and from the
    # second step NaN moments and weights -- the IEEE FP32 evaluation of the
    # step, on both sides.  NaNs compare equal whatever their bit patterns,
    # and must appear on exactly the same elements, only in those two blocks.
    n = 128 * 14
    w = W.custom("deg", [(n,)], "zip_sr")
    rng = np.random.default_rng(5)
    for recipe in ("zip_sr", "ze_eden", "factored", "torchao"):
        p = Pair(w.tensors, recipe)
        for t in range(1, 5):
            g = rng.normal(0, 1, n).astype(np.float32)
            g[0:128] = 0.0                                  # zero block
            g[128:256] *= 1e-38                             # subnormal moments
            g[256:384] *= 1e-25
            g[384:512] *= 1e15                              # huge, g^2 still finite
            g[512:640] = np.where(rng.random(128) < 0.5, 0.0, g[512:640] * 1e-3)
            g[640:768] *= np.float32(10.0) ** rng.uniform(-30, 10, 128).astype(np.float32)
            g[768:896] *= 1e25                              # every g^2 overflows
            g[896:1024] *= np.where(np.arange(128) % 2 == 0, 1e25, 1e-3).astype(np.float32)   # half of them
            g[1024:] *= 1e-3
            gt = torch.from_numpy(g).to(torch.bfloat16)
            p.step(t, [gt], seed=t)
            _assert_exact(p.compare(nan_ok=True), (recipe, t))
            th_g = p.gpu.view(0, "param").cpu().numpy()
            th_o = p.ora[0].param
            assert np.array_equal(np.isnan(th_g), np.isnan(th_o)), (recipe, t)
            assert not np.isnan(th_o[:768]).any() and not np.isnan(th_o[1024:]).any(), (recipe, t)
            if t == 1:
                assert not np.isnan(th_o).any()
                vs = p.gpu.view(0, "v_scale").cpu().numpy()
                assert np.isnan(vs[6]) if recipe == "ze_eden" else vs[6] == np.inf, (recipe, vs[6])


@pytest.mark.parametrize("recipe,flags", [("zip_sr", 0), ("zip_sr", q4.Q4_LM_HEAD_SR_ACTIVE), ("ze_eden", 0),
                                          ("torchao", 0), ("factored", 0)])
def test_empty_tensors_in_the_list(recipe, flags):
    # zero-size tensors first, in the middle and last (two flagged as the LM
    # head), around ragged and full ones: the chunk walk skips them and the
    # two-launch splits put them in either group
    shapes = [(0,), (300,), (0,), (64, 130), (0,), (1000,), (0,)]
    fl = [W.T_LM_HEAD, W.T_LM_HEAD, 0, W.T_FACTORED, 0, 0, W.T_LM_HEAD]
    w = W.custom("empty", shapes, recipe, flags=fl, grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, recipe)
    for t in range(1, 4):
        p.step(t, grads_for(w, t), seed=6, flags=flags)
        r = p.compare(exact_theta=recipe != "factored")
        assert r["codes"] == 0 and r["scales"] == 0 and r["theta"] == 0 and r["bf16"] == 0 and r["rc"] == 0, (t, r)
    assert p.gpu.status() == 0


def test_all_empty_list_is_a_no_op():
    w = W.custom("allempty", [(0,), (0,)], "zip_sr")
    st = q4.Q4State(w.tensors, "zip_sr")
    st.init()
    st.step(1, 1e-3, 0.9, 0.999, 1e-8, 0.1, flags=q4.Q4_LM_HEAD_SR_ACTIVE, max_grad_norm=1.0)
    torch.cuda.synchronize()
    assert st.status() == 0 and float(st.sqnorm.cpu()[0]) == 0.0


def test_factored_small_list():
    shapes = [(64, 96), (96,), (130, 128), (1, 256), (300, 40), (17,), (33, 64)]
    w = W.custom("fac", shapes, "factored", grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, "factored")
    for t in range(1, 11):
        p.step(t, grads_for(w, t))
        r = p.compare(exact_theta=False)
        assert r["codes"] == 0 and r["scales"] == 0, (t, r)
        assert r["rc"] == 0 and r["theta"] == 0 and r["bf16"] == 0, (t, r)


def test_factored_wide_rows():
    # rows of at least 256 columns take the vector path with the kernel's
    # incremental (row, column) tracking: widths that are multiples of 256,
    # and 1000 / 264 (multiples of 8 only), whose tiles straddle rows
    shapes = [(5, 256), (3, 768), (70, 512), (41, 1000), (9, 264), (300,), (2, 2048), (1, 4096)]
    w = W.custom("facwide", shapes, "factored", grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, "factored")
    for t in range(1, 7):
        p.step(t, grads_for(w, t))
        r = p.compare(exact_theta=False)
        assert r["codes"] == 0 and r["scales"] == 0, (t, r)
        assert r["rc"] == 0 and r["theta"] == 0 and r["bf16"] == 0, (t, r)


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "torchao"])
def test_sharded_tensor_matches_whole(recipe):
    # Two block-aligned shards with elem_offset produce the bits of the whole
    # tensor (the draws are keyed by the global element index; EDEN and the
    # scales are block-local), LM-head SR included.
    n, cut = 128 * 9 + 31, 128 * 4
    w = W.custom("shard", [(n,)], recipe, flags=[W.T_LM_HEAD])
    th = W.init_param(w.tensors[0], 0)
    whole = Pair(w.tensors, recipe, theta0=[th], tensor_ids=[4])
    parts = W.custom("shard2", [(cut,), (n - cut,)], recipe, flags=[W.T_LM_HEAD, W.T_LM_HEAD])
    split = Pair(parts.tensors, recipe, theta0=[th[:cut], th[cut:]], tensor_ids=[4, 4], elem_offsets=[0, cut])
    for t in range(1, 5):
        g = W.draw_grad(w, w.tensors[0], 0, t)
        whole.step(t, [g], seed=9, flags=1)
        split.step(t, [g[:cut], g[cut:]], seed=9, flags=1)
        for name in ("param", "param_bf16", "m_codes", "v_codes", "m_scale", "v_scale"):
            a = whole.gpu.view(0, name).cpu()
            b = torch.cat([split.gpu.view(0, name).cpu(), split.gpu.view(1, name).cpu()])
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (recipe, t, name)


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "factored", "torchao"])
def test_dequant_state_matches_oracle(recipe):
    shapes = [(40, 64), (200,), (3, 129)]
    w = W.custom("dq", shapes, recipe)
    p = Pair(w.tensors, recipe)
    for t in range(1, 4):
        p.step(t, grads_for(w, t))
    for i, o in enumerate(p.ora):
        m, v = p.gpu.dequant(i)
        torch.cuda.synchronize()
        assert np.array_equal(m.cpu().numpy(), o.m_dequant(recipe))
        vo = o.v_dequant(recipe)
        if o.factored:
            assert np.allclose(v.cpu().numpy(), vo, rtol=3e-5, atol=0)
        else:
            assert np.array_equal(v.cpu().numpy(), vo)


def test_state_init_header_and_zero_state():
    w = W.custom("hdr", [(300,), (64, 64)], "factored")
    p = Pair(w.tensors, "factored")
    h = p.gpu.header
    assert h.magic == 0x57413451 and h.format == 1 and h.recipe == 2 and h.block == 128
    assert h.n_tensors == 2 and h.numel_total == 300 + 64 * 64
    for name in ("m_codes", "m_scale"):
        assert int(getattr(p.gpu, name).abs().sum()) == 0


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "torchao"])
def test_m_sr_all_variant(recipe):
    # Rounding variant: State-SR for every tensor's first moment (flag 0x2).
    w = W.custom("msr", RAGGED, recipe, flags=[0] * len(RAGGED), grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, recipe)
    for t in range(1, 6):
        p.step(t, grads_for(w, t), seed=11, flags=q4.Q4_M_SR_ALL)
        _assert_exact(p.compare(), t)


def test_v_update_rtn_variant():
    # Rounding variant: Update-RTN in place of ZIP-SR's Update-SR (flag 0x4),
    # with mixed-magnitude gradients so that both neighbours occur.
    shapes = [(4096,), (300,), (64, 130)]
    w = W.custom("urtn", shapes, "zip_sr", flags=[W.T_LM_HEAD, 0, 0], grad="tensor_scaled", sigma=(1e-6, 1e-2))
    p = Pair(w.tensors, "zip_sr")
    for t in range(1, 8):
        p.step(t, grads_for(w, t), seed=2, flags=q4.Q4_V_UPDATE_RTN | q4.Q4_LM_HEAD_SR_ACTIVE)
        _assert_exact(p.compare(), t)


@pytest.mark.parametrize("urtn", [False, True])
@pytest.mark.parametrize("beta2", [0.999, 0.5])
def test_v_next_r_variant(urtn, beta2):
    # Rounding variant: ZIP-SR's Update rule in the next step's zero-gradient
    # preconditioner (flag 0x8), alone and with Update-RTN; beta2 = 0.5 moves
    # r' far from the same-step r.  Full tiles, ragged tails, LM-head SR.
    shapes = [(4096,), (300,), (64, 130), (128 * 13 + 17,), (2, 1024)]
    w = W.custom("nextr", shapes, "zip_sr", flags=[W.T_LM_HEAD, 0, 0, 0, 0], grad="tensor_scaled",
                 sigma=(1e-6, 1e-2))
    p = Pair(w.tensors, "zip_sr")
    hyper = dict(HYPER, beta2=beta2)
    flags = q4.Q4_V_NEXT_R | q4.Q4_LM_HEAD_SR_ACTIVE | (q4.Q4_V_UPDATE_RTN if urtn else 0)
    for t in range(1, 7):
        p.step(t, grads_for(w, t), seed=4, flags=flags, hyper=hyper)
        _assert_exact(p.compare(), t)


def test_torchao_mixed_magnitudes_every_sdyn4_rung():
    # |m'|/s spread over four decades inside each block, so every SDyn4
    # threshold (0.00275 .. 0.94375 of the scale, both signs) decides codes on
    # the fast path; plus ragged tails and a zero block.
    n = 128 * 40 + 77
    w = W.custom("taomix", [(n,), (3, 129)], "torchao")
    rng = np.random.default_rng(8)
    p = Pair(w.tensors, "torchao")
    for t in range(1, 9):
        gs = []
        for s in w.tensors:
            g = rng.normal(0, 1, s.numel) * 10.0 ** rng.uniform(-4, 0, s.numel)
            if s.numel == n:
                g[:128] = 0.0
            gs.append(torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16))
        p.step(t, gs, seed=t)
        _assert_exact(p.compare(), t)


def test_torchao_tensor_scaled_multistep():
    # The TorchAO baseline on a GPT-like list with per-tensor gradient scales in
    # [1e-5, 1e-2], LM head flagged and the final phase active (stays RTN).
    shapes = [(512, 256), (256,), (768, 256), (256,), (1000,)]
    flags = [W.T_LM_HEAD, 0, 0, 0, 0]
    w = W.custom("tao", shapes, "torchao", flags=flags, grad="tensor_scaled", sigma=(1e-5, 1e-2))
    p = Pair(w.tensors, "torchao")
    for t in range(9001, 9011):
        p.step(t, grads_for(w, t), seed=3, flags=q4.Q4_LM_HEAD_SR_ACTIVE)
        _assert_exact(p.compare(), t)
