"""ctypes binding of the q4adamw C ABI (include/q4adamw.h).

Argument marshalling only: every step of the optimizer runs in the CUDA
library.  Loading fails loudly when the built library is missing; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libq4adamw.so")

Q4_OK = 0
Q4_EINVAL = -1
Q4_EALIGN = -2
Q4_ESHAPE = -3
Q4_ERECIPE = -4
Q4_EVERSION = -5
Q4_ECUDA = -6
Q4_EWORKSPACE = -7

RECIPES = {"zip_sr": 0, "ze_eden": 1, "factored": 2, "torchao": 3}
Q4_T_LM_HEAD = 0x1
Q4_T_FACTORED = 0x2
Q4_LM_HEAD_SR_ACTIVE = 0x1
Q4_M_SR_ALL = 0x2
Q4_V_UPDATE_RTN = 0x4
Q4_V_NEXT_R = 0x8
Q4_STATUS_STAGE_TIMEOUT = 0x1
BLOCK = 128
NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024


class Q4Tensor(ctypes.Structure):
    """q4adamw_tensor_t."""
    _fields_ = [
        ("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("param_bf16", ctypes.c_void_p),
        ("m_codes", ctypes.c_void_p), ("m_scale", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("v_row", ctypes.c_void_p), ("v_col", ctypes.c_void_p),
        ("numel", ctypes.c_int64), ("rows", ctypes.c_int64), ("elem_offset", ctypes.c_uint64),
        ("tensor_id", ctypes.c_uint32), ("flags", ctypes.c_uint32),
    ]


class Q4Header(ctypes.Structure):
    """q4adamw_header_t."""
    _fields_ = [("magic", ctypes.c_uint32), ("format", ctypes.c_uint32), ("recipe", ctypes.c_uint32),
                ("block", ctypes.c_uint32), ("n_tensors", ctypes.c_int64), ("numel_total", ctypes.c_int64)]


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().q4adamw_strerror(status).decode()
        if status == Q4_ECUDA:
            msg += f" (cudaError {lib().q4adamw_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [{status}]")


_lib = None

EXPORTS = ("q4adamw_version", "q4adamw_strerror", "q4adamw_last_cuda_error", "q4adamw_state_bytes",
           "q4adamw_workspace_bytes", "q4adamw_state_init", "q4adamw_header_check", "q4adamw_step",
           "q4adamw_dequant_state", "q4adamw_codebook", "q4adamw_step_noalloc", "q4adamw_step_status",
           "q4adamw_grad_sqnorm", "q4adamw_step_clip", "q4adamw_draws", "q4adamw_set_stage_wait_limit",
           "q4adamw_step_noalloc_status", "q4adamw_dp_state_init", "q4adamw_dp_sums_floats",
           "q4adamw_dp_workspace_bytes",
           "q4adamw_dp_factored_sums", "q4adamw_dp_step", "q4adamw_grad_nonfinite")


def lib():
    """Load libq4adamw.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"q4adamw CUDA library not built: {LIB_PATH} is missing "
                          "(python -m bit_quantized_adamw_q4adamw_b300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, I64, U32, U64, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64,
                              ctypes.c_float)
    TP = ctypes.POINTER(Q4Tensor)
    L.q4adamw_version.restype = I
    L.q4adamw_strerror.argtypes = [I]
    L.q4adamw_strerror.restype = ctypes.c_char_p
    L.q4adamw_last_cuda_error.restype = I
    L.q4adamw_state_bytes.argtypes = [TP, I, I, P, P, P]
    L.q4adamw_workspace_bytes.argtypes = [TP, I, I, P]
    L.q4adamw_state_init.argtypes = [TP, I, I, ctypes.POINTER(Q4Header), P]
    L.q4adamw_header_check.argtypes = [ctypes.POINTER(Q4Header), I]
    L.q4adamw_step.argtypes = [TP, I, F, F, F, F, F, I64, U64, I, U32, P, I64, P]
    L.q4adamw_dequant_state.argtypes = [TP, I, P, P, P]
    L.q4adamw_step_noalloc.argtypes = [TP, I, F, F, F, F, F, I64, U64, I, U32, P]
    L.q4adamw_codebook.argtypes = [I, P, P]
    L.q4adamw_step_status.argtypes = [P, ctypes.POINTER(U32), P]
    L.q4adamw_grad_sqnorm.argtypes = [TP, I, P, P, I64, P]
    L.q4adamw_step_clip.argtypes = [TP, I, F, F, F, F, F, I64, U64, I, U32, F, P, P, I64, P]
    L.q4adamw_draws.argtypes = [U64, I64, U32, U64, U32, I64, P, P]
    L.q4adamw_set_stage_wait_limit.argtypes = [I64]
    L.q4adamw_step_noalloc_status.argtypes = [ctypes.POINTER(U32), P]
    L.q4adamw_dp_state_init.argtypes = [TP, I, I, P, ctypes.POINTER(Q4Header), P]
    L.q4adamw_dp_sums_floats.argtypes = [TP, I, I, P, P]
    L.q4adamw_dp_workspace_bytes.argtypes = [TP, I, I, P, P]
    L.q4adamw_dp_factored_sums.argtypes = [TP, I, I, P, F, P, P, P, I64, P]
    L.q4adamw_dp_step.argtypes = [TP, I, F, F, F, F, F, I64, U64, I, U32, P, P, F, P, P, I64, P]
    L.q4adamw_grad_nonfinite.argtypes = [TP, I, P, P, I64, P]
    for name in ("q4adamw_state_bytes", "q4adamw_workspace_bytes", "q4adamw_state_init", "q4adamw_header_check",
                 "q4adamw_step", "q4adamw_dequant_state", "q4adamw_codebook", "q4adamw_step_noalloc",
                 "q4adamw_step_status", "q4adamw_grad_sqnorm", "q4adamw_step_clip", "q4adamw_draws",
                 "q4adamw_set_stage_wait_limit", "q4adamw_step_noalloc_status", "q4adamw_dp_state_init",
                 "q4adamw_dp_sums_floats",
                 "q4adamw_dp_workspace_bytes", "q4adamw_dp_factored_sums", "q4adamw_dp_step",
                 "q4adamw_grad_nonfinite"):
        getattr(L, name).restype = I
    _lib = L
    return L
