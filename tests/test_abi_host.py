"""Host-side tests of the C ABI: the library loads, exports every symbol the
header declares, validates arguments without touching a GPU, sizes the state
as the pages state, and builds its codebooks bit-identical to the oracle's
independent construction."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import bit_quantized_adamw_q4adamw_b300 as q4
from bit_quantized_adamw_q4adamw_b300 import _native
from bit_quantized_adamw_q4adamw_b300.build import build
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4adamw.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q4adamw_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 10
    L = _native.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_native.EXPORTS)


def test_version_and_strerror():
    assert q4.q4adamw_version() == 1
    for st in range(-7, 1):
        s = q4.q4adamw_strerror(st)
        assert isinstance(s, str) and s
    assert q4.q4adamw_strerror(-99) == "unknown status"


@pytest.mark.parametrize("which,name", [(0, "nf4"), (1, "dyn4"), (2, "dyn4nz"), (3, "sdyn4"), (4, "lin4nz")])
def test_library_codebooks_match_oracle_bitwise(which, name):
    lv, th = q4.q4adamw_codebook(which)
    cb = O.codebooks()
    assert np.array_equal(lv.view(np.uint32), cb[name].view(np.uint32))
    assert np.array_equal(th.view(np.uint32), cb[name + "_t"].view(np.uint32))
    with pytest.raises(q4.Q4Error):
        q4.q4adamw_codebook(5)


def _t(numel, rows=1, flags=0, **kw):
    d = q4.Q4Tensor()
    d.numel = numel
    d.rows = rows
    d.flags = flags
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_state_bytes_is_1p0625_per_param():
    ts = [_t(128 * 1000), _t(4096), _t(2048 * 2048, 2048, q4.Q4_T_FACTORED)]
    n = sum(t.numel for t in ts)
    for recipe in ("zip_sr", "ze_eden"):
        q, s, tot = q4.q4adamw_state_bytes(ts, recipe)
        assert q == n and s == n // 16 and tot / n == 1.0625
        assert round(8 / (tot / n), 2) == 7.53
    q, s, tot = q4.q4adamw_state_bytes(ts, "factored")
    nf = 2048 * 2048
    assert q == (n - nf) + nf // 2
    assert s == (n - nf) // 16 + (nf // 128) * 4 + (2048 + 2048) * 4


def test_host_validation_errors():
    L = _native.lib()
    one = (q4.Q4Tensor * 1)(_t(256))
    assert L.q4adamw_state_bytes(one, 1, 7, None, None, None) == _native.Q4_ERECIPE
    assert L.q4adamw_state_bytes(one, -1, 0, None, None, None) == _native.Q4_EINVAL
    bad = (q4.Q4Tensor * 1)(_t(-5))
    assert L.q4adamw_state_bytes(bad, 1, 0, None, None, None) == _native.Q4_ESHAPE
    off = (q4.Q4Tensor * 1)(_t(256, elem_offset=64))
    assert L.q4adamw_state_bytes(off, 1, 0, None, None, None) == _native.Q4_ESHAPE
    fac = (q4.Q4Tensor * 1)(_t(1000, rows=7, flags=q4.Q4_T_FACTORED))
    assert L.q4adamw_state_bytes(fac, 1, 2, None, None, None) == _native.Q4_ESHAPE
    assert L.q4adamw_state_bytes(fac, 1, 0, None, None, None) == _native.Q4_OK   # flag ignored
    b = ctypes.c_int64()
    assert L.q4adamw_workspace_bytes(one, 1, 0, ctypes.byref(b)) == _native.Q4_OK and b.value % 256 == 0


def _valid_fake_tensor(numel=256):
    # Addresses are never dereferenced by validation; 256-aligned fakes.
    base = 1 << 40
    return _t(numel, param=base, grad=base + 0x10000, param_bf16=base + 0x20000, m_codes=base + 0x30000,
              m_scale=base + 0x40000, v_codes=base + 0x50000, v_scale=base + 0x60000)


def test_step_validation_happens_before_any_device_work():
    L = _native.lib()
    ws = ctypes.c_void_p(1 << 41)
    arr = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    args = dict(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.1, step=1, seed=0, recipe=0, flags=0)

    def call(arr=arr, n=1, ws=ws, wsb=1 << 20, **kw):
        a = dict(args, **kw)
        return L.q4adamw_step(arr, n, a["lr"], a["b1"], a["b2"], a["eps"], a["wd"], a["step"], a["seed"],
                              a["recipe"], a["flags"], ws, wsb, None)

    assert call(recipe=9) == _native.Q4_ERECIPE
    assert call(flags=0x10) == _native.Q4_EINVAL                      # unknown flag bit
    assert call(recipe=1, flags=_native.Q4_V_UPDATE_RTN) == _native.Q4_EINVAL   # ZIP-SR only
    assert call(recipe=1, flags=_native.Q4_V_NEXT_R) == _native.Q4_EINVAL       # ZIP-SR only
    assert call(recipe=3, flags=_native.Q4_V_NEXT_R) == _native.Q4_EINVAL
    assert call(step=0) == _native.Q4_EINVAL
    assert call(b1=1.0) == _native.Q4_EINVAL
    assert call(b2=-0.1) == _native.Q4_EINVAL
    assert call(eps=0.0) == _native.Q4_EINVAL
    assert call(lr=float("nan")) == _native.Q4_EINVAL
    assert call(n=-1) == _native.Q4_EINVAL
    assert call(ws=ctypes.c_void_p(0)) == _native.Q4_EWORKSPACE
    assert call(ws=ctypes.c_void_p((1 << 41) + 16)) == _native.Q4_EWORKSPACE
    assert call(wsb=16) == _native.Q4_EWORKSPACE
    mis = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    mis[0].param = mis[0].param + 4
    assert call(arr=mis) == _native.Q4_EALIGN
    nul = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    nul[0].v_codes = 0
    assert call(arr=nul) == _native.Q4_EINVAL
    nog = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    nog[0].grad = 0
    assert call(arr=nog) == _native.Q4_EINVAL


def test_clip_entry_points_validate_before_any_device_work():
    L = _native.lib()
    ws = ctypes.c_void_p(1 << 41)
    arr = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    sq = ctypes.c_void_p((1 << 41) + (1 << 30))

    def clip(max_norm=1.0, sqnorm=sq, arr=arr, flags=0, wsb=1 << 20):
        return L.q4adamw_step_clip(arr, 1, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 0, 0, flags, max_norm, sqnorm, ws, wsb,
                                   None)

    assert clip(max_norm=0.0) == _native.Q4_EINVAL
    assert clip(max_norm=-1.0) == _native.Q4_EINVAL
    assert clip(max_norm=float("nan")) == _native.Q4_EINVAL
    assert clip(max_norm=float("inf")) == _native.Q4_EINVAL
    assert clip(sqnorm=ctypes.c_void_p(0)) == _native.Q4_EINVAL
    assert clip(sqnorm=ctypes.c_void_p((1 << 41) + 2)) == _native.Q4_EALIGN
    assert clip(flags=0x10) == _native.Q4_EINVAL
    assert clip(wsb=16) == _native.Q4_EWORKSPACE

    def norm(arr=arr, n=1, out=sq, ws=ws, wsb=1 << 20):
        return L.q4adamw_grad_sqnorm(arr, n, out, ws, wsb, None)

    assert norm(out=ctypes.c_void_p(0)) == _native.Q4_EINVAL
    assert norm(out=ctypes.c_void_p((1 << 41) + 1)) == _native.Q4_EALIGN
    assert norm(n=-1) == _native.Q4_EINVAL
    assert norm(ws=ctypes.c_void_p(0)) == _native.Q4_EWORKSPACE
    assert norm(ws=ctypes.c_void_p((1 << 41) + 16)) == _native.Q4_EWORKSPACE
    assert norm(wsb=16) == _native.Q4_EWORKSPACE
    mis = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    mis[0].grad = mis[0].grad + 2
    assert norm(arr=mis) == _native.Q4_EALIGN
    nog = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    nog[0].grad = 0
    assert norm(arr=nog) == _native.Q4_EINVAL
    neg = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    neg[0].numel = -1
    assert norm(arr=neg) == _native.Q4_ESHAPE


def test_plain_c_client_compiles_links_and_runs(tmp_path):
    # the ABI from plain C99 (no Python, no torch): header, linking, host calls
    import os
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib = _native.LIB_PATH
    exe = str(tmp_path / "abi_c_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(root, "include"), os.path.join(root, "tests", "csrc", "abi_c_check.c"),
                    "-o", exe, lib, "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    env = dict(os.environ)
    import torch as _t
    env["LD_LIBRARY_PATH"] = os.pathsep.join([os.path.join(os.path.dirname(_t.__file__), "lib"),
                                              env.get("LD_LIBRARY_PATH", "")])
    out = subprocess.run([exe], capture_output=True, text=True, env=env)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr


def test_draws_validation_before_any_device_work():
    L = _native.lib()
    out = ctypes.c_void_p(1 << 41)
    assert L.q4adamw_draws(0, 1, 0, 0, 0, -1, out, None) == _native.Q4_EINVAL
    assert L.q4adamw_draws(0, 1, 0, 0, 0, 8, ctypes.c_void_p(0), None) == _native.Q4_EINVAL
    assert L.q4adamw_draws(0, 0, 0, 0, 0, 8, out, None) == _native.Q4_EINVAL           # step < 1
    assert L.q4adamw_draws(0, 2 ** 32, 0, 0, 0, 8, out, None) == _native.Q4_EINVAL     # step >= 2^32
    assert L.q4adamw_draws(0, 1, 0, 0, 16, 8, out, None) == _native.Q4_EINVAL          # purpose > 15
    assert L.q4adamw_draws(0, 1, 0, 0, 0, 8, ctypes.c_void_p((1 << 41) + 2), None) == _native.Q4_EALIGN
    assert L.q4adamw_draws(0, 1, 0, 0, 0, 0, ctypes.c_void_p(0), None) == 0            # nothing to do


def test_workspace_covers_the_norm_partials():
    # one huge tensor: few descriptors, many 2048-tile chunk partials
    L = _native.lib()
    n = ctypes.c_int64()
    big = (q4.Q4Tensor * 1)(_t(1 << 34, rows=1))
    assert L.q4adamw_workspace_bytes(big, 1, 0, ctypes.byref(n)) == 0
    chunks = (1 << 34) // (256 * 2048)
    assert n.value >= chunks * 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_step_without_gpu_fails_loudly():
    # No CPU fallback: a well-formed call on a machine without a GPU is a CUDA error.
    L = _native.lib()
    arr = (q4.Q4Tensor * 1)(_valid_fake_tensor())
    rc = L.q4adamw_step(arr, 1, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 0, 0, 0, ctypes.c_void_p(1 << 41), 1 << 20, None)
    assert rc == _native.Q4_ECUDA
    assert L.q4adamw_last_cuda_error() != 0


def test_header_check():
    h = q4.Q4Header(magic=0x57413451, format=1, recipe=0, block=128, n_tensors=1, numel_total=10)
    q4.q4adamw_header_check(h, "zip_sr")
    with pytest.raises(q4.Q4Error):
        q4.q4adamw_header_check(h, "ze_eden")
    h.format = 0
    with pytest.raises(q4.Q4Error):
        q4.q4adamw_header_check(h, "zip_sr")


def _dp_list(shards, full, rows, flags):
    arr = (q4.Q4Tensor * len(shards))()
    fake = 1 << 40                        # host-only calls never touch the pointers
    for k, ((start, n), r, f) in enumerate(zip(shards, rows, flags)):
        d = arr[k]
        d.param = d.grad = d.m_codes = d.m_scale = d.v_codes = d.v_scale = d.v_row = d.v_col = fake
        d.numel, d.rows, d.elem_offset, d.flags = n, r, start, f
    return arr, (ctypes.c_int64 * len(full))(*full)


def test_dp_host_calls_size_and_validate_shards():
    L = _native.lib()
    F = _native.Q4_T_FACTORED
    # a 100 x 200 parameter cut inside a row, an empty shard of a 48 x 256 one,
    # and a 1-D tensor (no statistics)
    arr, full = _dp_list([(8960, 11040), (0, 0), (128, 172)], [20000, 12288, 300], [100, 48, 1], [F, F, 0])
    n = ctypes.c_int64()
    assert L.q4adamw_dp_sums_floats(arr, 3, 2, full, ctypes.byref(n)) == 0
    assert n.value == (100 + 200) + (48 + 256)
    ws = ctypes.c_int64()
    assert L.q4adamw_dp_workspace_bytes(arr, 3, 2, full, ctypes.byref(ws)) == 0 and ws.value % 256 == 0
    # other recipes keep no statistics
    assert L.q4adamw_dp_sums_floats(arr, 3, 0, full, ctypes.byref(n)) == 0 and n.value == 0
    # NULL full_numel: whole tensors; the cut shard is then not a whole matrix
    assert L.q4adamw_dp_sums_floats(arr, 3, 2, None, ctypes.byref(n)) == _native.Q4_ESHAPE
    # the parameter's element count must be a multiple of rows, the shard inside it
    bad, full_bad = _dp_list([(0, 256)], [20001], [100], [F])
    assert L.q4adamw_dp_sums_floats(bad, 1, 2, full_bad, ctypes.byref(n)) == _native.Q4_ESHAPE
    out, full_out = _dp_list([(19968, 128)], [20000], [100], [F])
    assert L.q4adamw_dp_sums_floats(out, 1, 2, full_out, ctypes.byref(n)) == _native.Q4_ESHAPE
    # an empty factored shard still needs R and C (every rank updates them)
    empty, full_e = _dp_list([(0, 0)], [12288], [48], [F])
    empty[0].v_row = 0
    assert L.q4adamw_dp_sums_floats(empty, 1, 2, full_e, ctypes.byref(n)) == _native.Q4_EINVAL
    # device calls validate before any device work
    assert L.q4adamw_dp_step(arr, 3, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1, 0, 2, 0, full, None, 1.0, None, None, 0,
                             None) == _native.Q4_EWORKSPACE
    assert L.q4adamw_dp_factored_sums(arr, 3, 2, full, 1.0, None, None, None, 0, None) == _native.Q4_EINVAL
