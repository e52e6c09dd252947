"""CPU oracle for the fused 4-bit AdamW step -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and its
``--impl reference`` arm) may import this module.  The product path never
does; it has no CPU fallback.

The arithmetic lives in q4_oracle.c (plain C, single thread, FP32 with
``-ffp-contract=off``) and codebooks.py (levels built from their
definitions).  This file only compiles the C, marshals numpy arrays and keeps
per-tensor state between steps.

What pins each function (tests under tests/test_oracle_*.py):
  * Philox4x32-10 -- cuRAND's host Philox4_32_10 generator on the same
    (counter, key).
  * NF4 -- the same construction through scipy.special.ndtri (a different
    inverse-normal routine); structural facts (-1, 0, +1 exact; 16 distinct
    ascending levels).
  * Dyn4 / Dyn4-NZ -- exact rational definition (fractions.Fraction):
    every FP32 level is the nearest float to its rational value; 0 in Dyn4,
    none in Dyn4-NZ.  The level VALUES themselves are a reading (the pages
    print none): parity unpinned by the pages for the values.
  * RTN / State-SR / Update-RTN / Update-SR -- the near-zero-cell closed
    forms of the listing page's Table 1 by Monte Carlo; unbiasedness of
    State-SR in v and of Update-SR (ZIP-SR) in r; brute-force nearest level
    for RTN; |x - Q_SR| >= |x - Q_RTN| pointwise.
  * AdamW core -- with quantisation removed, torch.optim.AdamW (FP32 CPU)
    and a float64 numpy closed form.
  * ZE-EDEN scale -- the closed form |y|^2 / <y, yhat> in float64; exactly
    1 on blocks that sit on codebook levels.
  * Factored v -- brute-force float64 row/column means; rank-1 exactness;
    the weights against a float64 restatement of vhat = R_i C_j / mean(R);
    data-parallel shards (partial sums added over the shards, then the
    sums-based step) equal the whole-tensor step bit for bit when the sums
    are exact, and the partial sums equal brute-force float64 sums.
  * Gradient-norm clipping -- the sum of squares against textbook recursive
    pairwise summation (numpy, level by level) and a float64 error bound;
    the factor against torch.nn.utils.clip_grad_norm_ on exact-norm cases;
    the clipped step against the plain step on exactly pre-scaled gradients.
  * Storage -- 1.0625 bytes/param and 8 / 1.0625 = 7.53x, the figures the
    news page (paragraph 4) prints.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

from . import codebooks as _cb

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q4_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

BLOCK = 128
RECIPES = {"zip_sr": 0, "ze_eden": 1, "factored": 2, "torchao": 3}
T_LM_HEAD = 1
T_FACTORED = 2
LM_HEAD_SR_ACTIVE = 1
M_SR_ALL = 2          # State-SR for the first moment of every tensor (ablation)
V_UPDATE_RTN = 4      # Update-RTN instead of Update-SR under ZIP-SR (ablation)
V_NEXT_R = 8          # ZIP-SR rounds in the next step's zero-gradient preconditioner (ablation)
PURPOSE_M_SR = 0
PURPOSE_V_SR = 1
RULES = {"state_rtn": 0, "state_sr": 1, "update_rtn": 2, "update_sr": 3}


def build(force: bool = False) -> str:
    """Compile q4_oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC)):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class _Tensor(ctypes.Structure):
    _fields_ = [
        ("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("param_bf16", ctypes.c_void_p),
        ("m_codes", ctypes.c_void_p), ("m_scale", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("v_row", ctypes.c_void_p), ("v_col", ctypes.c_void_p),
        ("numel", ctypes.c_int64), ("rows", ctypes.c_int64),
        ("elem_offset", ctypes.c_uint64),
        ("tensor_id", ctypes.c_uint32), ("flags", ctypes.c_uint32),
    ]


class _Codebooks(ctypes.Structure):
    _fields_ = [
        ("nf4", ctypes.c_float * 16), ("nf4_t", ctypes.c_float * 15),
        ("dyn4", ctypes.c_float * 16), ("dyn4_t", ctypes.c_float * 15),
        ("dyn4nz", ctypes.c_float * 16), ("dyn4nz_t", ctypes.c_float * 15),
        ("sdyn4", ctypes.c_float * 16), ("sdyn4_t", ctypes.c_float * 15),
        ("lin4nz", ctypes.c_float * 16), ("lin4nz_t", ctypes.c_float * 15),
    ]


_lib = None
_cbs = None


def lib():
    global _lib
    if _lib is None:
        # Q4_ORACLE_LIB: a prebuilt oracle library to load instead (the mutation
        # tests point it at copies of q4_oracle.c with a planted mistake)
        L = ctypes.CDLL(os.environ.get("Q4_ORACLE_LIB") or build())
        P, U32, U64, I64, F = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, ctypes.c_float
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_draw.argtypes = [U64, U32, U32, U64, U32]
        L.oracle_draw.restype = U32
        L.oracle_draws.argtypes = [U64, U32, U32, U64, U32, I64, P]
        L.oracle_uniform.argtypes = [U32]
        L.oracle_uniform.restype = F
        L.oracle_host_scalars.argtypes = [F, F, F, F, I64, P]
        L.oracle_quant_block.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, F, F, P]
        L.oracle_quant_block.restype = F
        L.oracle_quant_block_r.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, F, F, F, P]
        L.oracle_quant_block_r.restype = F
        L.oracle_eden_scale.argtypes = [P, P, ctypes.c_int, P, F]
        L.oracle_eden_scale.restype = F
        L.oracle_dequant.argtypes = [P, P, P, I64, P]
        L.oracle_adamw_fp32.argtypes = [P, P, P, P, I64, F, F, F, F, F, I64]
        L.oracle_step_tensor.argtypes = [P, P, F, F, F, F, F, I64, U64, ctypes.c_int, U32]
        L.oracle_step_tensor.restype = ctypes.c_int
        L.oracle_step_tensor_clip.argtypes = [P, P, F, F, F, F, F, I64, U64, ctypes.c_int, U32, F]
        L.oracle_step_tensor_clip.restype = ctypes.c_int
        L.oracle_factored_partials.argtypes = [P, I64, F, P, P]
        L.oracle_step_tensor_sums.argtypes = [P, P, I64, P, P, F, F, F, F, F, I64, U64, ctypes.c_int, U32, F]
        L.oracle_step_tensor_sums.restype = ctypes.c_int
        L.oracle_grad_sqnorm.argtypes = [P, ctypes.c_int, P]
        L.oracle_grad_sqnorm.restype = F
        L.oracle_clip_factor.argtypes = [F, F]
        L.oracle_clip_factor.restype = F
        L.oracle_bf16_round.argtypes = [P, I64, P]
        _lib = L
    return _lib


def codebooks() -> dict:
    global _cbs
    if _cbs is None:
        _cbs = _cb.all_codebooks()
    return _cbs


def _cb_struct() -> _Codebooks:
    c = codebooks()
    s = _Codebooks()
    for name in ("nf4", "nf4_t", "dyn4", "dyn4_t", "dyn4nz", "dyn4nz_t", "sdyn4", "sdyn4_t", "lin4nz", "lin4nz_t"):
        getattr(s, name)[:] = [float(x) for x in c[name]]
    return s


def _ptr(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------- primitives
def philox(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def draws(seed: int, step: int, tensor_id: int, idx0: int, n: int, purpose: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.uint32)
    lib().oracle_draws(seed, step, tensor_id, idx0, purpose, n, _ptr(out))
    return out


def uniform(words: np.ndarray) -> np.ndarray:
    """u = (w >> 8) * 2^-24, the oracle's uniform (vectorised restatement)."""
    return ((np.asarray(words, dtype=np.uint32) >> 8).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def host_scalars(lr, beta1, beta2, weight_decay, step) -> dict:
    out = np.zeros(6, dtype=np.float32)
    lib().oracle_host_scalars(lr, beta1, beta2, weight_decay, step, _ptr(out))
    return dict(zip(("bc1", "c2", "step_size", "decay", "omb1", "omb2"), out.tolist()))


def quant_block(levels, thresholds, x, rule: str, words=None, c2=1.0, eps=1e-8, rbeta=None):
    """Quantise one block (len <= 128) with one of the four Table 1 rules.
    The Update rules round in r(x) = 1/(sqrt(x) c2 + eps), or with rbeta in
    r(x) = 1/(sqrt(rbeta x) c2 + eps) (the next-step variant: rbeta = beta2,
    c2 of step t+1)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.size
    assert n <= BLOCK
    L = np.ascontiguousarray(levels, dtype=np.float32)
    t = np.ascontiguousarray(thresholds, dtype=np.float32)
    w = np.zeros(max(n, 1), np.uint32) if words is None else np.ascontiguousarray(words, dtype=np.uint32)
    codes = np.zeros(max(n, 1), dtype=np.uint8)
    if rbeta is None:
        s = lib().oracle_quant_block(_ptr(L), _ptr(t), _ptr(x), n, RULES[rule], _ptr(w), c2, eps, _ptr(codes))
    else:
        s = lib().oracle_quant_block_r(_ptr(L), _ptr(t), _ptr(x), n, RULES[rule], _ptr(w), rbeta, c2, eps,
                                       _ptr(codes))
    return codes[:n], np.float32(s)


def eden_scale(v, codes, levels, s) -> np.float32:
    v = np.ascontiguousarray(v, dtype=np.float32)
    q = np.ascontiguousarray(codes, dtype=np.uint8)
    L = np.ascontiguousarray(levels, dtype=np.float32)
    return np.float32(lib().oracle_eden_scale(_ptr(v), _ptr(q), v.size, _ptr(L), np.float32(s)))


def dequant(levels, packed, scales, numel) -> np.ndarray:
    L = np.ascontiguousarray(levels, dtype=np.float32)
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.zeros(numel, dtype=np.float32)
    lib().oracle_dequant(_ptr(L), _ptr(p), _ptr(s), numel, _ptr(out))
    return out


def adamw_fp32(theta, grad, m, v, lr, beta1, beta2, eps, wd, step):
    """One unquantised FP32 AdamW step in place (numpy float32 arrays)."""
    for a in (theta, grad, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    lib().oracle_adamw_fp32(_ptr(theta), _ptr(grad), _ptr(m), _ptr(v), theta.size, lr, beta1, beta2, eps, wd, step)


def bf16_round(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(x.size, dtype=np.uint16)
    lib().oracle_bf16_round(_ptr(x), x.size, _ptr(out))
    return out


# ------------------------------------------------- gradient-norm clipping
def grad_sqnorm(grads) -> np.float32:
    """Sum of squares of a list of BF16 gradients (uint16 bit arrays) in the
    canonical FP32 order of q4_oracle.c (tile butterfly, per-tensor pairwise
    tree over tiles, tensors left to right)."""
    gs = [np.ascontiguousarray(g, dtype=np.uint16).reshape(-1) for g in grads]
    arr = (_Tensor * max(1, len(gs)))()
    for i, g in enumerate(gs):
        arr[i].grad = _ptr(g)
        arr[i].numel = g.size
    tiles = max([1] + [(g.size + 255) // 256 for g in gs])
    scratch = np.zeros(tiles, np.float32)
    return np.float32(lib().oracle_grad_sqnorm(ctypes.addressof(arr), len(gs), _ptr(scratch)))


def clip_factor(sqnorm, max_norm) -> np.float32:
    """min(1, max_norm / (sqrt(sqnorm) + 1e-6)) in FP32."""
    return np.float32(lib().oracle_clip_factor(np.float32(sqnorm), np.float32(max_norm)))


# ---------------------------------------------------------------- state
def nblocks(numel: int) -> int:
    return (numel + BLOCK - 1) // BLOCK


@dataclass
class OracleTensor:
    """Host copy of one parameter and its 4-bit state, as the oracle keeps it."""
    param: np.ndarray                 # float32 [numel]
    tensor_id: int
    rows: int = 1
    flags: int = 0
    elem_offset: int = 0
    factored: bool = False            # rank >= 2 under the factored recipe
    param_bf16: np.ndarray = None
    m_codes: np.ndarray = None
    m_scale: np.ndarray = None
    v_codes: np.ndarray = None
    v_scale: np.ndarray = None
    v_row: np.ndarray = None
    v_col: np.ndarray = None
    cols: int = None                  # a shard's parameter column count (None: whole tensor)
    _keep: list = field(default_factory=list)

    @classmethod
    def zeros_state(cls, param: np.ndarray, tensor_id: int, rows: int = 1, flags: int = 0,
                    elem_offset: int = 0, recipe: str = "zip_sr", cols: int | None = None) -> "OracleTensor":
        """cols: for one data-parallel shard of a factored parameter, the
        parameter's column count (its [rows, cols] matrix holds the shard's
        elements from elem_offset on); None for a whole tensor."""
        p = np.ascontiguousarray(param, dtype=np.float32).copy()
        n = p.size
        nb = nblocks(n)
        factored = recipe == "factored" and bool(flags & T_FACTORED)
        t = cls(param=p, tensor_id=tensor_id, rows=rows, flags=flags, elem_offset=elem_offset,
                factored=factored)
        t.cols = cols
        t.param_bf16 = np.zeros(n, np.uint16)
        t.m_codes = np.zeros(nb * BLOCK // 2, np.uint8)
        t.m_scale = np.zeros(nb, np.float32)
        if factored:
            t.v_row = np.zeros(rows, np.float32)
            t.v_col = np.zeros(n // rows if cols is None else cols, np.float32)
        else:
            t.v_codes = np.zeros(nb * BLOCK // 2, np.uint8)
            t.v_scale = np.zeros(nb, np.float32)
        return t

    def _desc(self, g) -> _Tensor:
        d = _Tensor()
        d.param = _ptr(self.param)
        d.grad = _ptr(g)
        d.param_bf16 = _ptr(self.param_bf16)
        d.m_codes = _ptr(self.m_codes)
        d.m_scale = _ptr(self.m_scale)
        d.v_codes = _ptr(self.v_codes)
        d.v_scale = _ptr(self.v_scale)
        d.v_row = _ptr(self.v_row)
        d.v_col = _ptr(self.v_col)
        d.numel = self.param.size
        d.rows = self.rows
        d.elem_offset = self.elem_offset
        d.tensor_id = self.tensor_id
        d.flags = self.flags
        return d

    def factored_partials(self, grad_bf16: np.ndarray, clip: float | None = None):
        """This shard's sums of (clip g)^2 per row and per column of the
        parameter's matrix (float64 arrays of rows and cols entries)."""
        assert self.factored
        g = np.ascontiguousarray(grad_bf16, dtype=np.uint16)
        cols = self.cols if self.cols is not None else self.param.size // self.rows
        rs = np.zeros(self.rows, np.float64)
        cs = np.zeros(cols, np.float64)
        d = self._desc(g)
        lib().oracle_factored_partials(ctypes.addressof(d), cols, 1.0 if clip is None else clip, _ptr(rs), _ptr(cs))
        return rs, cs

    def step_sums(self, grad_bf16: np.ndarray, row_sums, col_sums, lr, beta1, beta2, eps, wd, step, seed,
                  recipe: str, call_flags: int = 0, clip: float | None = None) -> None:
        """One step of this shard with the factored statistics taken from the
        sums over all shards (a tensor that is not factored steps as step())."""
        g = np.ascontiguousarray(grad_bf16, dtype=np.uint16)
        assert g.size == self.param.size
        cols = self.cols if self.cols is not None else self.param.size // self.rows
        rs = np.ascontiguousarray(row_sums, np.float64)
        cs = np.ascontiguousarray(col_sums, np.float64)
        assert not self.factored or (rs.size == self.rows and cs.size == cols)
        d = self._desc(g)
        cbs = _cb_struct()            # kept alive across the call
        rc = lib().oracle_step_tensor_sums(ctypes.addressof(cbs), ctypes.addressof(d), cols, _ptr(rs),
                                           _ptr(cs), lr, beta1, beta2, eps, wd, step, seed, RECIPES[recipe],
                                           call_flags, 1.0 if clip is None else clip)
        if rc != 0:
            raise ValueError(f"oracle_step_tensor_sums failed: {rc}")

    def step(self, grad_bf16: np.ndarray, lr, beta1, beta2, eps, wd, step, seed, recipe: str,
             call_flags: int = 0, clip: float | None = None) -> None:
        """One step; ``clip`` (a clip_factor() value) scales every gradient."""
        g = np.ascontiguousarray(grad_bf16, dtype=np.uint16)
        assert g.size == self.param.size
        assert self.cols is None, "a shard of a factored parameter steps with step_sums()"
        d = _Tensor()
        d.param = _ptr(self.param)
        d.grad = _ptr(g)
        d.param_bf16 = _ptr(self.param_bf16)
        d.m_codes = _ptr(self.m_codes)
        d.m_scale = _ptr(self.m_scale)
        d.v_codes = _ptr(self.v_codes)
        d.v_scale = _ptr(self.v_scale)
        d.v_row = _ptr(self.v_row)
        d.v_col = _ptr(self.v_col)
        d.numel = self.param.size
        d.rows = self.rows
        d.elem_offset = self.elem_offset
        d.tensor_id = self.tensor_id
        d.flags = self.flags
        cbs = _cb_struct()
        if clip is None:
            rc = lib().oracle_step_tensor(ctypes.addressof(cbs), ctypes.addressof(d), lr, beta1, beta2, eps, wd,
                                          step, seed, RECIPES[recipe], call_flags)
        else:
            rc = lib().oracle_step_tensor_clip(ctypes.addressof(cbs), ctypes.addressof(d), lr, beta1, beta2, eps,
                                               wd, step, seed, RECIPES[recipe], call_flags, clip)
        if rc != 0:
            raise ValueError(f"oracle_step_tensor failed: {rc}")

    def m_dequant(self, recipe: str = "zip_sr") -> np.ndarray:
        L = codebooks()["sdyn4" if recipe == "torchao" else "nf4"]
        return dequant(L, self.m_codes, self.m_scale, self.param.size)

    def v_dequant(self, recipe: str) -> np.ndarray:
        if self.factored:
            cols = self.param.size // self.rows
            rbar = np.float32(np.mean(self.v_row.astype(np.float64)))
            if rbar == 0:
                return np.zeros(self.param.size, np.float32)
            return ((self.v_row[:, None] * self.v_col[None, :]) / rbar).astype(np.float32).reshape(-1)
        L = codebooks()["dyn4" if recipe == "zip_sr" else "lin4nz" if recipe == "torchao" else "dyn4nz"]
        return dequant(L, self.v_codes, self.v_scale, self.param.size)
