"""q4adamw_step_noalloc: the step for callers that cannot allocate a workspace.

Some callers cannot give the library device memory for its workspace: they run
inside another framework's memory budget, or on a path where cudaMalloc's
implicit synchronisation is not acceptable.  q4adamw_step_noalloc serves them
from a fixed static device array.  These tests call it through the C ABI and
check, over two calls in a row, that it produces the same bits as
q4adamw_step with a caller workspace (the parity bar of every GPU test here is
bit-exact), that the status word in the static array reads 0 after each call
(q4adamw_step_noalloc_status), and that a tensor list too large for the static
array is refused.
This file is collected last on purpose.
"""

import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import _native
from bit_quantized_adamw_q4adamw_b300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [(4096,), (3, 200), (129,), (64, 128), (1000,)]
FLAGS = [0, W.T_LM_HEAD | W.T_FACTORED, 0, W.T_LM_HEAD | W.T_FACTORED, 0]


def _state(recipe):
    w = W.custom("na", SHAPES, recipe, flags=FLAGS)
    st = q4.Q4State(w.tensors, recipe)
    for i, s in enumerate(w.tensors):
        st.view(i, "param").copy_(W.init_param(s, i, device="cuda"))
    st.init()
    return w, st


def _buffers(st):
    names = ["param", "param_bf16", "m_codes", "m_scale", "v_codes", "v_scale", "v_row", "v_col"]
    return {n: getattr(st, n).clone() for n in names}


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "factored"])
def test_noalloc_matches_workspace_step_two_calls(recipe):
    w, ref = _state(recipe)
    _, na = _state(recipe)
    h = W.HYPER
    for t in (1, 2):
        for i, s in enumerate(w.tensors):
            g = W.draw_grad(w, s, i, t, device="cuda")
            ref.view(i, "grad").copy_(g)
            na.view(i, "grad").copy_(g)
        ref.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=5,
                 flags=q4.Q4_LM_HEAD_SR_ACTIVE)
        q4.q4adamw_step_noalloc(na.descs, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t, 5,
                                recipe, q4.Q4_LM_HEAD_SR_ACTIVE)
        torch.cuda.synchronize()
        # the static scratch's status word: the noalloc step ran to completion
        assert q4.q4adamw_step_noalloc_status() == 0, (recipe, t)
        a, b = _buffers(ref), _buffers(na)
        for name in a:
            assert torch.equal(a[name].view(torch.uint8), b[name].view(torch.uint8)), (recipe, t, name)


def test_noalloc_rejects_lists_beyond_its_scratch():
    # 40000 one-block tensors need more than the 4 MiB static scratch for their
    # descriptors alone: refused before any device work (pointers are never used).
    n = 40000
    arr = (q4.Q4Tensor * n)()
    base = 1 << 40
    for k in range(n):
        d = arr[k]
        d.param, d.grad, d.m_codes, d.m_scale = base, base, base, base
        d.v_codes, d.v_scale, d.numel, d.rows = base, base, 128, 1
    assert q4.q4adamw_workspace_bytes(arr, "zip_sr") > _native.NOALLOC_SCRATCH_BYTES
    rc = _native.lib().q4adamw_step_noalloc(arr, n, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 0, 0, 0, None)
    assert rc == _native.Q4_EWORKSPACE
