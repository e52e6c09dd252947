"""B300-native fused 4-bit AdamW optimizer step (ZIP-SR / ZE-EDEN).

Python binding of the C ABI in include/q4adamw.h.  The functions below carry
the C names and only marshal arguments (torch tensors -> device pointers,
streams -> handles); every step of the optimizer runs in the CUDA library
(bit_quantized_adamw_q4adamw_b300/_build/libq4adamw.so).  ``Q4State`` is a
convenience holder that allocates the state buffers with torch for a list of
parameters laid out in flat arenas.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _native
from ._native import (BLOCK, Q4_LM_HEAD_SR_ACTIVE, Q4_M_SR_ALL, Q4_T_FACTORED, Q4_T_LM_HEAD, Q4_V_NEXT_R,
                      Q4_V_UPDATE_RTN,
                      RECIPES, Q4Error, Q4Header,
                      Q4Tensor, lib)

__all__ = ["q4adamw_version", "q4adamw_strerror", "q4adamw_state_bytes", "q4adamw_workspace_bytes",
           "q4adamw_state_init", "q4adamw_header_check", "q4adamw_step", "q4adamw_step_noalloc",
           "q4adamw_dequant_state", "q4adamw_step_status", "q4adamw_grad_sqnorm", "q4adamw_step_clip", "q4adamw_draws",
           "q4adamw_codebook", "q4adamw_set_stage_wait_limit", "q4adamw_step_noalloc_status",
           "q4adamw_grad_nonfinite", "Q4State", "Q4Tensor", "Q4Header", "Q4Error", "RECIPES", "Q4_T_LM_HEAD",
           "Q4_T_FACTORED", "Q4_LM_HEAD_SR_ACTIVE", "Q4_M_SR_ALL", "Q4_V_UPDATE_RTN", "Q4_V_NEXT_R", "BLOCK"]


def _recipe(r) -> int:
    return RECIPES[r] if isinstance(r, str) else int(r)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _array(tensors):
    if isinstance(tensors, ctypes.Array):
        return tensors, len(tensors)
    arr = (Q4Tensor * len(tensors))(*tensors)
    return arr, len(tensors)


def _check(status: int, what: str):
    if status != _native.Q4_OK:
        raise Q4Error(status, what)


def q4adamw_version() -> int:
    return lib().q4adamw_version()


def q4adamw_strerror(status: int) -> str:
    return lib().q4adamw_strerror(status).decode()


def q4adamw_state_bytes(tensors, recipe):
    arr, n = _array(tensors)
    q, s, t = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().q4adamw_state_bytes(arr, n, _recipe(recipe), ctypes.byref(q), ctypes.byref(s), ctypes.byref(t)),
           "q4adamw_state_bytes")
    return q.value, s.value, t.value


def q4adamw_workspace_bytes(tensors, recipe) -> int:
    arr, n = _array(tensors)
    b = ctypes.c_int64()
    _check(lib().q4adamw_workspace_bytes(arr, n, _recipe(recipe), ctypes.byref(b)), "q4adamw_workspace_bytes")
    return b.value


def q4adamw_state_init(tensors, recipe, stream=None) -> Q4Header:
    arr, n = _array(tensors)
    h = Q4Header()
    _check(lib().q4adamw_state_init(arr, n, _recipe(recipe), ctypes.byref(h), _stream(stream)),
           "q4adamw_state_init")
    return h


def q4adamw_header_check(header: Q4Header, recipe) -> None:
    _check(lib().q4adamw_header_check(ctypes.byref(header), _recipe(recipe)), "q4adamw_header_check")


def q4adamw_step(tensors, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, workspace: torch.Tensor,
                 stream=None) -> None:
    arr, n = _array(tensors)
    _check(lib().q4adamw_step(arr, n, lr, beta1, beta2, eps, weight_decay, int(step), int(seed) & (2 ** 64 - 1),
                              _recipe(recipe), int(flags), ctypes.c_void_p(workspace.data_ptr()),
                              workspace.numel() * workspace.element_size(), _stream(stream)), "q4adamw_step")


def q4adamw_grad_sqnorm(tensors, out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Sum of squares of the BF16 gradients into out (a device float32 tensor
    of one element), in the library's fixed pairwise order."""
    assert out.dtype == torch.float32 and out.numel() >= 1 and out.is_cuda
    arr, n = _array(tensors)
    _check(lib().q4adamw_grad_sqnorm(arr, n, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "q4adamw_grad_sqnorm")


def q4adamw_step_clip(tensors, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags, max_grad_norm,
                      sqnorm: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """q4adamw_step with the gradients scaled by the global-norm clip factor
    min(1, max_grad_norm / (sqrt(sqnorm) + 1e-6)); sqnorm is a device float32."""
    assert sqnorm.dtype == torch.float32 and sqnorm.is_cuda
    arr, n = _array(tensors)
    _check(lib().q4adamw_step_clip(arr, n, lr, beta1, beta2, eps, weight_decay, int(step), int(seed) & (2 ** 64 - 1),
                                   _recipe(recipe), int(flags), float(max_grad_norm),
                                   ctypes.c_void_p(sqnorm.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "q4adamw_step_clip")


def q4adamw_draws(seed, step, tensor_id, idx0, purpose, out: torch.Tensor, stream=None) -> None:
    """The step's Philox words for elements idx0 .. idx0+out.numel()-1 into a
    device int32/uint32 tensor (purpose 0: m State-SR, 1: v Update-SR)."""
    assert out.is_cuda and out.element_size() == 4
    _check(lib().q4adamw_draws(int(seed) & (2 ** 64 - 1), int(step), int(tensor_id), int(idx0), int(purpose),
                               out.numel(), ctypes.c_void_p(out.data_ptr()), _stream(stream)), "q4adamw_draws")


def q4adamw_step_noalloc(tensors, lr, beta1, beta2, eps, weight_decay, step, seed, recipe, flags,
                         stream=None) -> None:
    """q4adamw_step using the library's fixed static device scratch instead of a
    workspace, for callers that cannot allocate one (see include/q4adamw.h)."""
    arr, n = _array(tensors)
    _check(lib().q4adamw_step_noalloc(arr, n, lr, beta1, beta2, eps, weight_decay, int(step),
                                      int(seed) & (2 ** 64 - 1), _recipe(recipe), int(flags), _stream(stream)),
           "q4adamw_step_noalloc")


def q4adamw_grad_nonfinite(tensors, out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Number of NaN / +-inf BF16 gradients of the list into out (a device int64
    tensor of one element)."""
    assert out.is_cuda and out.element_size() == 8 and out.numel() >= 1
    arr, n = _array(tensors)
    _check(lib().q4adamw_grad_nonfinite(arr, n, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "q4adamw_grad_nonfinite")


def q4adamw_step_noalloc_status(stream=None) -> int:
    """Status word of the last q4adamw_step_noalloc on the current device (0 =
    completed); synchronises the stream."""
    v = ctypes.c_uint32()
    _check(lib().q4adamw_step_noalloc_status(ctypes.byref(v), _stream(stream)), "q4adamw_step_noalloc_status")
    return v.value


def q4adamw_set_stage_wait_limit(cycles: int) -> None:
    """Per-thread limit (SM clock cycles) of the step kernel's wait for a staged
    tile; 0 restores the default (about one second)."""
    _check(lib().q4adamw_set_stage_wait_limit(int(cycles)), "q4adamw_set_stage_wait_limit")


def q4adamw_step_status(workspace: torch.Tensor, stream=None) -> int:
    """Status word of the last q4adamw_step on `workspace` (0 = completed);
    synchronises the stream."""
    v = ctypes.c_uint32()
    _check(lib().q4adamw_step_status(ctypes.c_void_p(workspace.data_ptr()), ctypes.byref(v), _stream(stream)),
           "q4adamw_step_status")
    return v.value


def q4adamw_dequant_state(tensor: Q4Tensor, recipe, m_out: torch.Tensor | None = None,
                          v_out: torch.Tensor | None = None, stream=None) -> None:
    _check(lib().q4adamw_dequant_state(ctypes.byref(tensor), _recipe(recipe),
                                       ctypes.c_void_p(m_out.data_ptr() if m_out is not None else 0),
                                       ctypes.c_void_p(v_out.data_ptr() if v_out is not None else 0),
                                       _stream(stream)), "q4adamw_dequant_state")


def q4adamw_codebook(which: int):
    lv = np.zeros(16, np.float32)
    th = np.zeros(15, np.float32)
    _check(lib().q4adamw_codebook(which, lv.ctypes.data, th.ctypes.data), "q4adamw_codebook")
    return lv, th


# --------------------------------------------------------------------------
@dataclass
class _Slot:
    numel: int
    rows: int
    flags: int
    tensor_id: int
    elem_offset: int
    off: int        # element offset in the param/grad/bf16 arenas
    boff: int       # block offset in the code/scale arenas
    roff: int = 0   # factored: offset in the row arena
    coff: int = 0   # factored: offset in the column arena


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


class Q4State:
    """Parameters, gradients and 4-bit state of a tensor list in flat device arenas.

    specs: sequence of (numel, rows, flags) or objects with .numel/.rows/.flags.
    Every tensor starts at a multiple of 128 elements in the arenas, which
    satisfies the library's alignment rules.
    """

    def __init__(self, specs, recipe, device="cuda", tensor_ids=None, elem_offsets=None, bf16_out=True):
        self.recipe = recipe
        self.device = torch.device(device)
        self.slots = []
        off = boff = roff = coff = 0
        for i, s in enumerate(specs):
            numel, rows, flags = (s.numel, s.rows, s.flags) if hasattr(s, "numel") else s
            tid = tensor_ids[i] if tensor_ids is not None else i
            eo = elem_offsets[i] if elem_offsets is not None else 0
            sl = _Slot(numel, rows, flags, tid, eo, off, boff)
            nb = (numel + BLOCK - 1) // BLOCK
            if self.is_factored(sl):
                sl.roff, sl.coff = roff, coff
                roff = _round_up(roff + rows, 4)
                coff = _round_up(coff + numel // rows, 4)
            self.slots.append(sl)
            off += nb * BLOCK
            boff += nb
        dev = self.device
        self.param = torch.zeros(max(off, 1), dtype=torch.float32, device=dev)
        self.grad = torch.zeros(max(off, 1), dtype=torch.bfloat16, device=dev)
        self.param_bf16 = torch.zeros(max(off, 1), dtype=torch.bfloat16, device=dev) if bf16_out else None
        self.m_codes = torch.zeros(max(boff, 1) * 64, dtype=torch.uint8, device=dev)
        self.m_scale = torch.zeros(max(boff, 1), dtype=torch.float32, device=dev)
        self.v_codes = torch.zeros(max(boff, 1) * 64, dtype=torch.uint8, device=dev)
        self.v_scale = torch.zeros(max(boff, 1), dtype=torch.float32, device=dev)
        self.v_row = torch.zeros(max(roff, 1), dtype=torch.float32, device=dev)
        self.v_col = torch.zeros(max(coff, 1), dtype=torch.float32, device=dev)
        self.descs = (Q4Tensor * len(self.slots))()
        for i, sl in enumerate(self.slots):
            self.descs[i] = self._desc(sl)
        self.workspace = torch.empty(max(q4adamw_workspace_bytes(self.descs, recipe), 256), dtype=torch.uint8,
                                     device=dev)
        self.sqnorm = torch.zeros(1, dtype=torch.float32, device=dev)
        self.header = None

    def is_factored(self, sl) -> bool:
        return self.recipe == "factored" and bool(sl.flags & Q4_T_FACTORED) and len_ok(sl)

    def _desc(self, sl: _Slot) -> Q4Tensor:
        f32, b16, u8 = 4, 2, 1
        d = Q4Tensor()
        d.param = self.param.data_ptr() + sl.off * f32
        d.grad = self.grad.data_ptr() + sl.off * b16
        d.param_bf16 = (self.param_bf16.data_ptr() + sl.off * b16) if self.param_bf16 is not None else 0
        d.m_codes = self.m_codes.data_ptr() + sl.boff * 64 * u8
        d.m_scale = self.m_scale.data_ptr() + sl.boff * f32
        if self.is_factored(sl):
            d.v_codes = 0
            d.v_scale = 0
            d.v_row = self.v_row.data_ptr() + sl.roff * f32
            d.v_col = self.v_col.data_ptr() + sl.coff * f32
        else:
            d.v_codes = self.v_codes.data_ptr() + sl.boff * 64 * u8
            d.v_scale = self.v_scale.data_ptr() + sl.boff * f32
            d.v_row = 0
            d.v_col = 0
        d.numel = sl.numel
        d.rows = sl.rows
        d.elem_offset = sl.elem_offset
        d.tensor_id = sl.tensor_id
        d.flags = sl.flags
        return d

    # views of one tensor's buffers
    def view(self, i: int, name: str) -> torch.Tensor:
        sl = self.slots[i]
        nb = (sl.numel + BLOCK - 1) // BLOCK
        if name in ("param", "grad", "param_bf16"):
            return getattr(self, name)[sl.off:sl.off + sl.numel]
        if name in ("m_codes", "v_codes"):
            return getattr(self, name)[sl.boff * 64:(sl.boff + nb) * 64]
        if name in ("m_scale", "v_scale"):
            return getattr(self, name)[sl.boff:sl.boff + nb]
        if name == "v_row":
            return self.v_row[sl.roff:sl.roff + sl.rows]
        if name == "v_col":
            return self.v_col[sl.coff:sl.coff + sl.numel // sl.rows]
        raise KeyError(name)

    def init(self, stream=None) -> Q4Header:
        self.header = q4adamw_state_init(self.descs, self.recipe, stream)
        return self.header

    def grad_sqnorm(self, stream=None) -> torch.Tensor:
        """Device float32 sum of squares of the gradient arena's tensors."""
        q4adamw_grad_sqnorm(self.descs, self.sqnorm, self.workspace, stream)
        return self.sqnorm

    def step(self, step, lr, beta1, beta2, eps, weight_decay, seed=0, flags=0, stream=None,
             max_grad_norm=None, sqnorm=None) -> None:
        """One fused step.  With max_grad_norm the gradients are clipped to that
        global 2-norm: the sum of squares is `sqnorm` (a device float32, e.g.
        all-reduced over data-parallel ranks) or, when None, computed here."""
        if max_grad_norm is None:
            q4adamw_step(self.descs, lr, beta1, beta2, eps, weight_decay, step, seed, self.recipe, flags,
                         self.workspace, stream)
            return
        if sqnorm is None:
            sqnorm = self.grad_sqnorm(stream)
        q4adamw_step_clip(self.descs, lr, beta1, beta2, eps, weight_decay, step, seed, self.recipe, flags,
                          max_grad_norm, sqnorm, self.workspace, stream)

    def status(self, stream=None) -> int:
        """Status word of the last step (0 = completed); synchronises."""
        return q4adamw_step_status(self.workspace, stream)

    def dequant(self, i: int, stream=None):
        sl = self.slots[i]
        m = torch.empty(sl.numel, dtype=torch.float32, device=self.device)
        v = torch.empty(sl.numel, dtype=torch.float32, device=self.device)
        q4adamw_dequant_state(self.descs[i], self.recipe, m, v, stream)
        return m, v

    @property
    def numel(self) -> int:
        return sum(s.numel for s in self.slots)


def len_ok(sl) -> bool:
    return sl.numel > 0 and sl.rows >= 1 and sl.numel % sl.rows == 0
