"""Global gradient-norm clipping on the GPU against the oracle.

q4adamw_grad_sqnorm must reproduce the oracle's FP32 sum of squares bit for
bit (both are recursive pairwise summation per tensor, tensors left to
right), at sizes that span the lane, tile, group, 2048-tile chunk and
multi-level chunk-tree stages, with ragged tails and empty tensors.
q4adamw_step_clip must then match the oracle's clipped step exactly (the
factored recipe at its stated tolerances).
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import workloads as W
from oracle import oracle as O
from parity_util import HYPER, Pair, bf16_bits, grads_for

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _gpu_sqnorm(grads):
    """grads: list of device bfloat16 tensors (16-B aligned)."""
    arr = (q4.Q4Tensor * max(1, len(grads)))()
    for i, g in enumerate(grads):
        arr[i].grad = g.data_ptr() if g.numel() > 0 else 0
        arr[i].numel = g.numel()
        arr[i].rows = 1
    L = q4.lib()
    nbytes = ctypes.c_int64()
    assert L.q4adamw_workspace_bytes(arr, len(grads), 0, ctypes.byref(nbytes)) == 0
    ws = torch.empty(max(nbytes.value, 256), dtype=torch.uint8, device=DEV)
    out = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
    rc = L.q4adamw_grad_sqnorm(arr, len(grads), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                               ws.numel(), None)
    assert rc == 0, q4.q4adamw_strerror(rc)
    torch.cuda.synchronize()
    return np.float32(out.cpu().numpy()[0])


def _device_bf16(x: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    # a fresh allocation is 256-B aligned
    return t.to(DEV)


def _check(gs):
    got = _gpu_sqnorm(gs)
    want = O.grad_sqnorm([bf16_bits(g) for g in gs])
    if np.isnan(want):
        assert np.isnan(got)
    else:
        assert got.view(np.uint32) == want.view(np.uint32), (got, want)
    return got


CHUNK = 2048 * 256


@pytest.mark.parametrize("sizes", [
    [1], [7], [8], [255], [256], [257], [8191], [8192 + 9],
    [CHUNK - 1], [CHUNK], [CHUNK + 1], [3 * CHUNK + 12345],
    [0, 17, 0, 256 * 33 + 5, 1],
    [128 * 13 + 17, 4096 + 64, 1000, 3 * 129, 257 * 7],
])
def test_sqnorm_bit_exact(sizes):
    rng = np.random.default_rng(len(sizes) * 1000 + sum(sizes) % 997)
    gs = [_device_bf16(rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 2, n)) for n in sizes]
    _check(gs)


def test_sqnorm_many_tensors():
    # more tensors than one pass of the final left-to-right sum (1024) holds
    rng = np.random.default_rng(11)
    sizes = rng.integers(0, 3000, size=1300)
    gs = [_device_bf16(rng.standard_normal(int(n)) * rng.uniform(1e-3, 3.0)) for n in sizes]
    _check(gs)


def test_sqnorm_multilevel_chunk_tree():
    # more than 512 chunks in one tensor: the per-tensor tree runs two levels
    n = 513 * CHUNK + 1000
    g = torch.randn(n, device=DEV, generator=torch.Generator(DEV).manual_seed(5)).to(torch.bfloat16)
    _check([g])
    del g
    torch.cuda.empty_cache()


def test_sqnorm_special_values():
    rng = np.random.default_rng(2)
    base = rng.standard_normal(5000).astype(np.float32)
    tiny = base * np.float32(1e-30)                 # squares underflow (subnormal or 0)
    huge = base.copy()
    huge[17] = 3e38                                 # square overflows to inf
    nan = base.copy()
    nan[4000] = np.nan
    assert np.isfinite(_check([_device_bf16(tiny)]))
    assert np.isinf(_check([_device_bf16(base), _device_bf16(huge)]))
    assert np.isnan(_check([_device_bf16(nan), _device_bf16(base)]))
    assert _check([_device_bf16(np.zeros(1000))]) == 0.0
    assert _check([]) == 0.0


RAGGED = [(1,), (5,), (127,), (128,), (129,), (255,), (256,), (1000,), (3, 129), (257, 7), (4096 + 64,),
          (7, 128), (128 * 13 + 17,)]


@pytest.mark.parametrize("recipe,flags", [("zip_sr", 0), ("zip_sr", q4.Q4_LM_HEAD_SR_ACTIVE), ("ze_eden", 0),
                                          ("ze_eden", q4.Q4_LM_HEAD_SR_ACTIVE), ("torchao", 0),
                                          ("zip_sr", q4.Q4_V_UPDATE_RTN), ("zip_sr", q4.Q4_M_SR_ALL)])
def test_clipped_step_bit_exact(recipe, flags):
    fl = [W.T_LM_HEAD if i % 4 == 0 else 0 for i in range(len(RAGGED))]
    w = W.custom("clip", RAGGED, recipe, flags=fl, grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, recipe)
    clips = []
    for t in range(1, 7):
        # the global norm here is about 0.2: 0.05 clips, 100 does not
        mgn = 0.05 if t % 3 else 100.0
        p.step(t, grads_for(w, t), seed=5, flags=flags, max_grad_norm=mgn)
        clips.append(p.last_clip)
        r = p.compare()
        assert r["codes"] == 0 and r["scales"] == 0 and r["theta"] == 0 and r["bf16"] == 0, (t, r)
    assert min(clips) < 0.5 and max(clips) == 1.0


def test_clipped_step_factored():
    shapes = [(64, 96), (96,), (130, 128), (1, 256), (300, 40), (17,), (33, 64)]
    w = W.custom("facclip", shapes, "factored", grad="normal", sigma=(1e-3, 1e-3))
    p = Pair(w.tensors, "factored")
    for t in range(1, 6):
        p.step(t, grads_for(w, t), max_grad_norm=0.03)
        assert p.last_clip < 1.0
        r = p.compare(exact_theta=False)
        assert r["codes"] == 0 and r["scales"] == 0, (t, r)
        assert r["rc"] == 0 and r["theta"] == 0 and r["bf16"] == 0, (t, r)


def test_clip_with_external_sqnorm():
    # a caller-supplied sum of squares (as after a data-parallel all-reduce)
    # is used as given: clip from 4x the local sum equals the oracle's factor
    w = W.custom("ext", [(1000,), (3, 129)], "zip_sr", grad="normal", sigma=(1e-2, 1e-2))
    p = Pair(w.tensors, "zip_sr")
    g = grads_for(w, 1)
    for i, x in enumerate(g):
        p.gpu.view(i, "grad").copy_(x)
    local = O.grad_sqnorm([bf16_bits(x) for x in g])
    total = np.float32(local * np.float32(4.0))
    sq = torch.tensor([float(total)], dtype=torch.float32, device=DEV)
    h = HYPER
    p.gpu.step(1, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0, 0, max_grad_norm=0.1, sqnorm=sq)
    clip = O.clip_factor(total, 0.1)
    for i, x in enumerate(g):
        p.ora[i].step(bf16_bits(x), h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 1, 0, "zip_sr",
                      0, clip=clip)
    torch.cuda.synchronize()
    r = p.compare()
    assert r["codes"] == 0 and r["theta"] == 0 and r["scales"] == 0, r
