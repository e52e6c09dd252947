"""Helpers for GPU-versus-oracle parity tests (test infrastructure).

Both sides start from the same seeded inputs (workloads.py draws them on the
CPU) and then evolve independently: the oracle keeps its own state; nothing
the CUDA library produces is ever fed to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import workloads as W
from oracle import oracle as O

HYPER = W.HYPER


def neq_f32(a: np.ndarray, b: np.ndarray, nan_ok: bool = False) -> np.ndarray:
    """Bitwise inequality of FP32 arrays.  With nan_ok, two NaNs count as
    equal whatever their bit patterns: IEEE 754 leaves a NaN result's sign
    and payload open, and the host and the GPU make different ones."""
    d = a.view(np.uint32) != b.view(np.uint32)
    return d & ~(np.isnan(a) & np.isnan(b)) if nan_ok else d


def neq_bf16(a: np.ndarray, b: np.ndarray, nan_ok: bool = False) -> np.ndarray:
    """Inequality of BF16 bit arrays; with nan_ok two NaNs count as equal."""
    d = a != b
    if nan_ok:
        isnan = lambda x: ((x & 0x7f80) == 0x7f80) & ((x & 0x7f) != 0)   # noqa: E731
        d &= ~(isnan(a) & isnan(b))
    return d


def bf16_close(a: np.ndarray, b: np.ndarray, theta_tol: float = 1e-6) -> np.ndarray:
    """BF16 copies of weights that agree within theta_tol * max(1, |theta|):
    equal up to one BF16 unit in the last place, or (near zero, where the two
    may round to opposite signs) within the weight tolerance itself."""
    fa = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fb = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d = np.abs(fa - fb)
    return (d <= 2.0 ** -7 * np.maximum(np.abs(fa), np.abs(fb))) | (d <= 2 * theta_tol * np.maximum(1.0, np.abs(fb)))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


class Pair:
    """A CUDA Q4State and the oracle's per-tensor state for the same tensor list."""

    def __init__(self, specs, recipe, *, tensor_ids=None, elem_offsets=None, theta0=None, seed_inputs=0):
        self.specs = list(specs)
        self.recipe = recipe
        n = len(self.specs)
        self.tids = list(tensor_ids) if tensor_ids is not None else list(range(n))
        self.offs = list(elem_offsets) if elem_offsets is not None else [0] * n
        self.gpu = q4.Q4State(self.specs, recipe, tensor_ids=self.tids, elem_offsets=self.offs)
        self.ora = []
        for i, s in enumerate(self.specs):
            th = theta0[i] if theta0 is not None else W.init_param(s, self.tids[i], "cpu", seed_inputs)
            th = th.numpy() if isinstance(th, torch.Tensor) else np.asarray(th, np.float32)
            self.gpu.view(i, "param").copy_(torch.from_numpy(th))
            self.ora.append(O.OracleTensor.zeros_state(th, self.tids[i], rows=s.rows, flags=s.flags,
                                                       elem_offset=self.offs[i], recipe=recipe))
        self.gpu.init()
        torch.cuda.synchronize()

    def step(self, t, grads, seed=0, flags=0, hyper=HYPER, max_grad_norm=None):
        """grads: list of CPU bfloat16 tensors (one per tensor).  With
        max_grad_norm both sides clip by the global norm; the GPU's sum of
        squares must then equal the oracle's bit for bit (asserted)."""
        for i, g in enumerate(grads):
            self.gpu.view(i, "grad").copy_(g)
        self.gpu.step(t, hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"], hyper["weight_decay"], seed,
                      flags, max_grad_norm=max_grad_norm)
        clip = None
        if max_grad_norm is not None:
            bits = [bf16_bits(g) for g in grads]
            sq = O.grad_sqnorm(bits)
            got = np.float32(self.gpu.sqnorm.cpu().numpy()[0])
            assert got.view(np.uint32) == sq.view(np.uint32), (t, got, sq)
            clip = O.clip_factor(sq, max_grad_norm)
            self.last_clip = float(clip)
        for i, g in enumerate(grads):
            self.ora[i].step(bf16_bits(g), hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                             hyper["weight_decay"], t, seed, self.recipe, flags, clip=clip)
        torch.cuda.synchronize()

    def compare(self, exact_theta=True, rc_rtol=1e-5, theta_tol=1e-6, nan_ok=False):
        """Element-by-element comparison; returns a dict of mismatch counts.
        nan_ok: NaN results on both sides count as equal (only where the
        step's IEEE FP32 evaluation makes NaNs, e.g. after an overflow)."""
        out = {"codes": 0, "scales": 0, "theta": 0, "bf16": 0, "rc": 0, "max_dtheta": 0.0}
        for i, o in enumerate(self.ora):
            s = self.specs[i]
            nb = O.nblocks(s.numel)
            mc = self.gpu.view(i, "m_codes").cpu().numpy()
            out["codes"] += int((mc != o.m_codes).sum())
            ms = self.gpu.view(i, "m_scale").cpu().numpy()
            out["scales"] += int(neq_f32(ms, o.m_scale, nan_ok).sum())
            if o.factored:
                R = self.gpu.view(i, "v_row").cpu().numpy().astype(np.float64)
                C = self.gpu.view(i, "v_col").cpu().numpy().astype(np.float64)
                out["rc"] += int((np.abs(R - o.v_row) > rc_rtol * np.abs(o.v_row)).sum())
                out["rc"] += int((np.abs(C - o.v_col) > rc_rtol * np.abs(o.v_col)).sum())
            else:
                vc = self.gpu.view(i, "v_codes").cpu().numpy()
                out["codes"] += int((vc != o.v_codes).sum())
                vs = self.gpu.view(i, "v_scale").cpu().numpy()
                out["scales"] += int(neq_f32(vs, o.v_scale, nan_ok).sum())
            th = self.gpu.view(i, "param").cpu().numpy()
            d = np.abs(th.astype(np.float64) - o.param)
            out["max_dtheta"] = max(out["max_dtheta"], float(d.max(initial=0.0)))
            if exact_theta:
                out["theta"] += int(neq_f32(th, o.param, nan_ok).sum())
            else:
                out["theta"] += int((d > theta_tol * np.maximum(1.0, np.abs(o.param))).sum())
            b16 = bf16_bits(self.gpu.view(i, "param_bf16"))
            if exact_theta:
                out["bf16"] += int(neq_bf16(b16, o.param_bf16, nan_ok).sum())
            else:
                out["bf16"] += int((~bf16_close(b16, o.param_bf16, theta_tol)).sum())
            assert nb == ms.size
        return out


def grads_for(w: W.Workload, t: int, seed=0, specs=None, tids=None):
    specs = specs or w.tensors
    tids = tids or list(range(len(specs)))
    return [W.draw_grad(w, s, tid, t, "cpu", seed) for s, tid in zip(specs, tids)]
