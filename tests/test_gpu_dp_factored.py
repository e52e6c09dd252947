"""Data-parallel shards of factored parameters on the GPU, through the C ABI.

AReno docs "4-bit AdamW", section "State representation": under data
parallelism each rank's row and column sums of g^2 are added over the group,
and R and C are updated from the totals.  The library's three-call protocol
(q4adamw_dp_factored_sums -> the caller adds the sums over the ranks ->
q4adamw_dp_step) is checked here on one GPU, with the ranks' buffers side by
side and their sums added on the device (the addition an all-reduce makes):

  * one rank holding whole tensors reproduces q4adamw_step bit for bit;
  * two ranks whose shards cut factored parameters inside rows (one rank
    holding no element of a parameter) match the oracle's shard steps --
    codes and scales bit for bit, R and C within 1e-5 relative, weights
    within 1e-6 max(1, |theta|) -- and every rank's copy of R and C is the
    same.
"""
import ctypes

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
RECIPE = q4.RECIPES["factored"]


def _i64(vals):
    return (ctypes.c_int64 * len(vals))(*vals)


class Rank:
    """One rank's shards: [(tensor index, start, numel)] over the parameters
    `specs`; each shard has its own parameter, gradient and state buffers and,
    for factored parameters, its own full-size R and C."""

    def __init__(self, specs, shards, flags):
        self.specs, self.shards = specs, shards
        self.arr = (q4.Q4Tensor * len(shards))()
        self.full = []
        self.bufs = []
        dev = "cuda"
        for k, (i, start, n) in enumerate(shards):
            s = specs[i]
            nb = (n + 127) // 128
            fact = bool(flags[i] & W.T_FACTORED)
            b = dict(param=torch.zeros(max(n, 1), dtype=torch.float32, device=dev),
                     grad=torch.zeros(max(n, 1), dtype=torch.bfloat16, device=dev),
                     bf16=torch.zeros(max(n, 1), dtype=torch.bfloat16, device=dev),
                     mc=torch.zeros(max(nb, 1) * 64, dtype=torch.uint8, device=dev),
                     ms=torch.zeros(max(nb, 1), dtype=torch.float32, device=dev))
            if fact:
                b["vrow"] = torch.zeros(s.rows, dtype=torch.float32, device=dev)
                b["vcol"] = torch.zeros(s.numel // s.rows, dtype=torch.float32, device=dev)
            else:
                b["vc"] = torch.zeros(max(nb, 1) * 64, dtype=torch.uint8, device=dev)
                b["vs"] = torch.zeros(max(nb, 1), dtype=torch.float32, device=dev)
            d = self.arr[k]
            d.param, d.grad, d.param_bf16 = b["param"].data_ptr(), b["grad"].data_ptr(), b["bf16"].data_ptr()
            d.m_codes, d.m_scale = b["mc"].data_ptr(), b["ms"].data_ptr()
            d.v_codes, d.v_scale = (0, 0) if fact else (b["vc"].data_ptr(), b["vs"].data_ptr())
            d.v_row, d.v_col = (b["vrow"].data_ptr(), b["vcol"].data_ptr()) if fact else (0, 0)
            d.numel, d.rows, d.elem_offset, d.tensor_id, d.flags = n, s.rows, start, i, flags[i]
            self.full.append(s.numel)
            self.bufs.append(b)
        self.full_arr = _i64(self.full)
        L = _native.lib()
        nf, wsb = ctypes.c_int64(), ctypes.c_int64()
        assert L.q4adamw_dp_sums_floats(self.arr, len(shards), RECIPE, self.full_arr, ctypes.byref(nf)) == 0
        assert L.q4adamw_dp_workspace_bytes(self.arr, len(shards), RECIPE, self.full_arr, ctypes.byref(wsb)) == 0
        self.sums = torch.zeros(max(nf.value, 1), dtype=torch.float32, device=dev)
        self.n_sums = nf.value
        self.ws = torch.empty(max(wsb.value, 256), dtype=torch.uint8, device=dev)
        h = q4.Q4Header()
        assert L.q4adamw_dp_state_init(self.arr, len(shards), RECIPE, self.full_arr, ctypes.byref(h), None) == 0

    def load(self, thetas):
        for (i, start, n), b in zip(self.shards, self.bufs):
            b["param"][:n].copy_(torch.from_numpy(thetas[i][start:start + n]))

    def set_grads(self, grads):
        for (i, start, n), b in zip(self.shards, self.bufs):
            b["grad"][:n].copy_(grads[i][start:start + n])

    def partial_sums(self):
        rc = _native.lib().q4adamw_dp_factored_sums(self.arr, len(self.shards), RECIPE, self.full_arr, 1.0, None,
                                                   ctypes.c_void_p(self.sums.data_ptr()),
                                                   ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(), None)
        assert rc == 0

    def step(self, t, total_sums, flags=0):
        rc = _native.lib().q4adamw_dp_step(self.arr, len(self.shards), H["lr"], H["beta1"], H["beta2"], H["eps"],
                                          H["weight_decay"], t, 21, RECIPE, flags, self.full_arr,
                                          ctypes.c_void_p(total_sums.data_ptr()), 1.0, None,
                                          ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(), None)
        assert rc == 0


SPECS = [(100, 200), (300,), (64, 264), (48, 256), (5, 40)]
FLAGS = [W.T_FACTORED, 0, W.T_FACTORED | W.T_LM_HEAD, W.T_FACTORED, W.T_FACTORED]


def _workload():
    return W.custom("dp", SPECS, "factored", flags=FLAGS, grad="normal", sigma=(1e-3, 1e-3))


def test_dp_single_rank_equals_the_step():
    w = _workload()
    specs = w.tensors
    thetas = [W.init_param(s, i).numpy() for i, s in enumerate(specs)]
    r = Rank(specs, [(i, 0, s.numel) for i, s in enumerate(specs)], FLAGS)
    r.load(thetas)
    st = q4.Q4State(specs, "factored")
    for i in range(len(specs)):
        st.view(i, "param").copy_(torch.from_numpy(thetas[i]))
    st.init()
    for t in range(1, 4):
        grads = [W.draw_grad(w, s, i, t) for i, s in enumerate(specs)]
        r.set_grads(grads)
        for i, g in enumerate(grads):
            st.view(i, "grad").copy_(g)
        r.partial_sums()
        r.step(t, r.sums, q4.Q4_LM_HEAD_SR_ACTIVE)
        st.step(t, H["lr"], H["beta1"], H["beta2"], H["eps"], H["weight_decay"], seed=21,
                flags=q4.Q4_LM_HEAD_SR_ACTIVE)
        torch.cuda.synchronize()
        for i, b in enumerate(r.bufs):
            n = specs[i].numel
            for name, view in (("param", "param"), ("bf16", "param_bf16"), ("mc", "m_codes"), ("ms", "m_scale"),
                               ("vrow", "v_row"), ("vcol", "v_col"), ("vc", "v_codes"), ("vs", "v_scale")):
                if name not in b:
                    continue
                a = b[name]
                if name in ("param", "bf16"):
                    a = a[:n]
                elif name in ("mc", "vc"):
                    a = a[:((n + 127) // 128) * 64]
                elif name in ("ms", "vs"):
                    a = a[:(n + 127) // 128]
                assert torch.equal(a.view(torch.uint8), st.view(i, view).contiguous().view(torch.uint8)), (t, i, name)


def _shards_for(specs, cuts):
    """cuts[i] = a (a multiple of 128): rank 0 holds [0, a) of tensor i,
    rank 1 [a, numel); a = numel leaves rank 1 an empty shard, a = 0 rank 0."""
    r0 = [(i, 0, cuts[i]) for i in range(len(specs))]
    r1 = [(i, cuts[i], specs[i].numel - cuts[i]) for i in range(len(specs))]
    return r0, r1


def test_dp_two_ranks_match_the_oracle_shard_steps():
    w = _workload()
    specs = w.tensors
    # 100 x 200 cut inside a row (128*70 = row 44, column 160); 64 x 264 cut
    # at a row boundary (128*33 = 16*264); 48 x 256 held by rank 0 only; 5 x 40
    # (one block) held by rank 1 only; the 1-D tensor split too
    cuts = [128 * 70, 128, 128 * 33, 48 * 256, 0]
    r0, r1 = _shards_for(specs, cuts)
    thetas = [W.init_param(s, i).numpy() for i, s in enumerate(specs)]
    ranks = [Rank(specs, r0, FLAGS), Rank(specs, r1, FLAGS)]
    for r in ranks:
        r.load(thetas)
    ora = []
    for shards in (r0, r1):
        row = []
        for i, start, n in shards:
            s = specs[i]
            fact = bool(FLAGS[i] & W.T_FACTORED)
            row.append(O.OracleTensor.zeros_state(thetas[i][start:start + n], i, rows=s.rows, flags=FLAGS[i],
                                                  elem_offset=start, recipe="factored",
                                                  cols=(s.numel // s.rows) if fact else None))
        ora.append(row)
    assert ranks[0].n_sums == ranks[1].n_sums == sum(s.rows + s.numel // s.rows for i, s in enumerate(specs)
                                                     if FLAGS[i] & W.T_FACTORED)
    for t in range(1, 5):
        grads = [W.draw_grad(w, s, i, t) for i, s in enumerate(specs)]
        for r in ranks:
            r.set_grads(grads)
            r.partial_sums()
        total = ranks[0].sums + ranks[1].sums           # the all-reduce
        for r in ranks:
            r.step(t, total, q4.Q4_LM_HEAD_SR_ACTIVE)
        # the oracle: float64 partial sums of every shard, added, then each shard's step
        sums = {}
        for shards, orow in zip((r0, r1), ora):
            for (i, start, n), o in zip(shards, orow):
                if o.factored:
                    rs, cs = o.factored_partials(bf16_bits(grads[i][start:start + n]))
                    if i in sums:
                        sums[i] = (sums[i][0] + rs, sums[i][1] + cs)
                    else:
                        sums[i] = (rs, cs)
        for shards, orow in zip((r0, r1), ora):
            for (i, start, n), o in zip(shards, orow):
                rs, cs = sums.get(i, (np.zeros(1), np.zeros(1)))
                o.step_sums(bf16_bits(grads[i][start:start + n]), rs, cs, H["lr"], H["beta1"], H["beta2"], H["eps"],
                            H["weight_decay"], t, 21, "factored", q4.Q4_LM_HEAD_SR_ACTIVE)
        torch.cuda.synchronize()
        for k, (r, orow) in enumerate(zip(ranks, ora)):
            for (i, start, n), b, o in zip(r.shards, r.bufs, orow):
                nb = (n + 127) // 128
                assert np.array_equal(b["mc"][:nb * 64].cpu().numpy(), o.m_codes), (t, k, i)
                assert not neq_f32(b["ms"][:nb].cpu().numpy(), o.m_scale).any(), (t, k, i)
                th = b["param"][:n].cpu().numpy()
                if o.factored:
                    R = b["vrow"].cpu().numpy().astype(np.float64)
                    C = b["vcol"].cpu().numpy().astype(np.float64)
                    assert (np.abs(R - o.v_row) <= 1e-5 * np.abs(o.v_row)).all(), (t, k, i)
                    assert (np.abs(C - o.v_col) <= 1e-5 * np.abs(o.v_col)).all(), (t, k, i)
                    d = np.abs(th.astype(np.float64) - o.param)
                    assert (d <= 1e-6 * np.maximum(1.0, np.abs(o.param))).all(), (t, k, i, float(d.max(initial=0)))
                    assert bf16_close(bf16_bits(b["bf16"][:n]), o.param_bf16).all(), (t, k, i)
                else:
                    assert not neq_f32(th, o.param).any(), (t, k, i)
                    assert np.array_equal(b["vc"][:nb * 64].cpu().numpy(), o.v_codes), (t, k, i)
        # every rank's R and C are the same bits
        for k in range(len(specs)):
            if FLAGS[k] & W.T_FACTORED:
                assert torch.equal(ranks[0].bufs[k]["vrow"], ranks[1].bufs[k]["vrow"]), (t, k)
                assert torch.equal(ranks[0].bufs[k]["vcol"], ranks[1].bufs[k]["vcol"]), (t, k)
