"""Failure detection of the step, exercised without faulting the GPU.

  * The step kernel's wait for a staged tile is bounded.  With the limit cut
    to one SM clock cycle (q4adamw_set_stage_wait_limit) and the L2 flushed
    just before, warps give up on data that is still on its way from HBM:
    the call returns, the status word reports Q4_STATUS_STAGE_TIMEOUT, every
    warp drains its own copies before it stops, and the next step with the
    default limit runs to completion and reports 0.  Nothing hangs: the
    copies always complete, only later.
  * Guard bands: every buffer the step writes (FP32 and BF16 weights, codes,
    scales, R, C and the workspace) sits between 256-byte canaries of a known
    pattern; after steps on a ragged tensor list in every recipe -- checked
    element by element against the oracle -- no canary byte has changed.
"""
import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import _native
from bit_quantized_adamw_q4adamw_b300 import workloads as W
from oracle import oracle as O
from parity_util import HYPER, bf16_bits, bf16_close, neq_f32

pytestmark = pytest.mark.gpu

H = HYPER


def _flush_l2():
    # a write four times the 126 MB L2: the step's inputs then come from HBM,
    # so a warp's first staged tile is still on its way at the first wait
    buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    torch.cuda.synchronize()


def _stepped_state(recipe="zip_sr"):
    w = W.custom("to", [(4_000_000,), (257, 10_000), (4096,)], recipe, grad="normal", sigma=(1e-3, 1e-3))
    st = q4.Q4State(w.tensors, recipe)
    for i, s in enumerate(w.tensors):
        st.view(i, "param").copy_(W.init_param(s, i, device="cuda"))
        st.view(i, "grad").copy_(W.draw_grad(w, s, i, 1, device="cuda"))
    st.init()
    return st


ATTEMPTS = 5   # each flushed; whether a given warp's data is still on its way at its first wait is timing


def test_stage_wait_timeout_sets_status_and_returns():
    st = _stepped_state()
    seen = []
    try:
        q4.q4adamw_set_stage_wait_limit(1)
        for k in range(ATTEMPTS):
            _flush_l2()
            st.step(1 + k, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"])
            seen.append(st.status())
            if seen[-1] & _native.Q4_STATUS_STAGE_TIMEOUT:
                break
        assert seen[-1] & _native.Q4_STATUS_STAGE_TIMEOUT, seen
        assert all(s in (0, _native.Q4_STATUS_STAGE_TIMEOUT) for s in seen), seen
    finally:
        q4.q4adamw_set_stage_wait_limit(0)
    # the context is intact: a step with the default limit completes
    st.step(ATTEMPTS + 1, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"])
    assert st.status() == 0
    assert torch.isfinite(st.param).all()


def test_stage_wait_timeout_through_the_noalloc_status():
    st = _stepped_state("ze_eden")
    seen = []
    try:
        q4.q4adamw_set_stage_wait_limit(1)
        for k in range(ATTEMPTS):
            _flush_l2()
            q4.q4adamw_step_noalloc(st.descs, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], 1 + k,
                                    0, "ze_eden", 0)
            seen.append(q4.q4adamw_step_noalloc_status())
            if seen[-1] & _native.Q4_STATUS_STAGE_TIMEOUT:
                break
        assert seen[-1] & _native.Q4_STATUS_STAGE_TIMEOUT, seen
    finally:
        q4.q4adamw_set_stage_wait_limit(0)
    q4.q4adamw_step_noalloc(st.descs, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], ATTEMPTS + 1,
                            0, "ze_eden", 0)
    assert q4.q4adamw_step_noalloc_status() == 0


# ------------------------------------------------------------------ guard bands
G = 256                       # canary bytes on each side (keeps 256-B alignment)
CANARY = 0xA5


class _Guarded:
    """One device allocation with a payload of `nbytes` between two canaries."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.buf = torch.full((G + max(self.n, 1) + G,), CANARY, dtype=torch.uint8, device="cuda")

    @property
    def ptr(self):
        return self.buf.data_ptr() + G

    def payload(self, dtype):
        return self.buf[G:G + self.n].view(dtype)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:G] == CANARY).all() and (b[G + self.n:] == CANARY).all())


SHAPES = [(1,), (5,), (127,), (129,), (255,), (3, 129), (257, 7), (1000,), (64, 130), (4096 + 64,)]


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden", "torchao", "factored"])
def test_guard_bands_intact_after_ragged_steps(recipe):
    fl = [W.T_LM_HEAD if i % 4 == 0 else 0 for i in range(len(SHAPES))]
    if recipe == "factored":
        fl = [f | (W.T_FACTORED if len(s) == 2 else 0) for f, s in zip(fl, SHAPES)]
    w = W.custom("guard", SHAPES, recipe, flags=fl, grad="normal", sigma=(1e-3, 1e-3))
    arr = (q4.Q4Tensor * len(w.tensors))()
    bufs, ora = [], []
    for i, s in enumerate(w.tensors):
        nb = (s.numel + 127) // 128
        fact = recipe == "factored" and bool(s.flags & W.T_FACTORED)
        b = dict(param=_Guarded(4 * s.numel), grad=_Guarded(2 * s.numel), bf16=_Guarded(2 * s.numel),
                 mc=_Guarded(64 * nb), ms=_Guarded(4 * nb))
        if fact:
            b.update(vrow=_Guarded(4 * s.rows), vcol=_Guarded(4 * (s.numel // s.rows)))
        else:
            b.update(vc=_Guarded(64 * nb), vs=_Guarded(4 * nb))
        th = W.init_param(s, i).numpy()
        b["param"].payload(torch.float32).copy_(torch.from_numpy(th))
        d = arr[i]
        d.param, d.grad, d.param_bf16 = b["param"].ptr, b["grad"].ptr, b["bf16"].ptr
        d.m_codes, d.m_scale = b["mc"].ptr, b["ms"].ptr
        d.v_codes, d.v_scale = (0, 0) if fact else (b["vc"].ptr, b["vs"].ptr)
        d.v_row, d.v_col = (b["vrow"].ptr, b["vcol"].ptr) if fact else (0, 0)
        d.numel, d.rows, d.elem_offset, d.tensor_id, d.flags = s.numel, s.rows, 0, i, s.flags
        bufs.append(b)
        ora.append(O.OracleTensor.zeros_state(th, i, rows=s.rows, flags=s.flags, recipe=recipe))
    ws = _Guarded(q4.q4adamw_workspace_bytes(arr, recipe))
    q4.q4adamw_state_init(arr, recipe)
    wsv = ws.buf[G:G + ws.n]
    for t in range(1, 4):
        grads = [W.draw_grad(w, s, i, t) for i, s in enumerate(w.tensors)]
        for i, g in enumerate(grads):
            bufs[i]["grad"].payload(torch.bfloat16).copy_(g)
        rc = _native.lib().q4adamw_step(arr, len(w.tensors), H["lr"], H["beta1"], H["beta2"], H["eps"],
                                        H["weight_decay"], t, 9, q4.RECIPES[recipe], q4.Q4_LM_HEAD_SR_ACTIVE,
                                        ws.ptr, ws.n, None)
        assert rc == 0
        for i, g in enumerate(grads):
            ora[i].step(bf16_bits(g), H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], t, 9, recipe,
                        q4.Q4_LM_HEAD_SR_ACTIVE)
        torch.cuda.synchronize()
        assert q4.q4adamw_step_status(wsv) == 0
        for i, (b, o) in enumerate(zip(bufs, ora)):
            for name, g in list(b.items()) + [("workspace", ws)]:
                assert g.intact(), (recipe, t, i, name)
            th = b["param"].payload(torch.float32).cpu().numpy()
            assert np.array_equal(b["mc"].payload(torch.uint8).cpu().numpy(), o.m_codes), (recipe, t, i)
            assert not neq_f32(b["ms"].payload(torch.float32).cpu().numpy(), o.m_scale).any(), (recipe, t, i)
            if o.factored:
                d = np.abs(th.astype(np.float64) - o.param)
                assert (d <= 1e-6 * np.maximum(1.0, np.abs(o.param))).all(), (recipe, t, i)
                assert bf16_close(bf16_bits(b["bf16"].payload(torch.bfloat16)), o.param_bf16).all()
            else:
                assert not neq_f32(th, o.param).any(), (recipe, t, i)
                assert np.array_equal(bf16_bits(b["bf16"].payload(torch.bfloat16)), o.param_bf16), (recipe, t, i)
                assert np.array_equal(b["vc"].payload(torch.uint8).cpu().numpy(), o.v_codes), (recipe, t, i)
                assert not neq_f32(b["vs"].payload(torch.float32).cpu().numpy(), o.v_scale).any(), (recipe, t, i)
