"""World-size-2 gloo tests of the multi-rank path on the CPU.

The step needs no collective: each rank steps its own block-aligned shards
(elem_offset = global start), and the union of the shards must equal the
single-rank result bit for bit.  The bench's max-over-ranks timing reduction
is exercised with the same process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_quantized_adamw_q4adamw_b300 import sharding
from bit_quantized_adamw_q4adamw_b300 import workloads as W

SHAPES = [(1000,), (37, 129), (4096,), (5,), (130, 64)]
FLAGS = [W.T_LM_HEAD, 0, 0, 0, W.T_LM_HEAD]


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _run_oracle(shards, recipe, steps):
    from oracle import oracle as O
    w = W.custom("mr", SHAPES, recipe, flags=FLAGS)
    h = W.HYPER
    outs = []
    for sh in shards:
        spec = w.tensors[sh.tensor]
        th = W.init_param(spec, sh.tensor).numpy()[sh.start:sh.start + sh.numel]
        t = O.OracleTensor.zeros_state(th, sh.tensor, flags=spec.flags, elem_offset=sh.elem_offset, recipe=recipe)
        for k in range(1, steps + 1):
            g = W.draw_grad(w, spec, sh.tensor, k)[sh.start:sh.start + sh.numel].contiguous()
            t.step(g.view(torch.int16).numpy().view(np.uint16), h["lr"], h["beta1"], h["beta2"], h["eps"],
                   h["weight_decay"], k, 11, recipe, O.LM_HEAD_SR_ACTIVE)
        outs.append((sh.tensor, sh.start, t.param.copy(), t.m_codes.copy(), t.v_codes.copy(), t.v_scale.copy()))
    return outs


def _worker(rank, world, port, recipe, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shards = sharding.partition([int(np.prod(s)) for s in SHAPES], world, rank)
        outs = _run_oracle(shards, recipe, steps=3)
        gathered = [None] * world
        dist.all_gather_object(gathered, outs)
        import bench
        mx = bench.max_over_ranks(float(rank + 1) * 10.0)
        if rank == 0:
            q.put((gathered, mx))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("recipe", ["zip_sr", "ze_eden"])
def test_two_rank_shards_equal_single_rank(recipe):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, recipe, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, mx = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert mx == 20.0
    whole = _run_oracle(sharding.partition([int(np.prod(s)) for s in SHAPES], 1, 0), recipe, steps=3)
    parts = {}
    for outs in gathered:
        for tensor, start, th, mc, vc, vs in outs:
            parts.setdefault(tensor, []).append((start, th, mc, vc, vs))
    for tensor, start, th, mc, vc, vs in whole:
        ps = sorted(parts[tensor], key=lambda x: x[0])
        assert ps[0][0] == 0
        assert np.array_equal(np.concatenate([p[1] for p in ps]), th)
        assert np.array_equal(np.concatenate([p[2] for p in ps]), mc)
        assert np.array_equal(np.concatenate([p[3] for p in ps]), vc)
        assert np.array_equal(np.concatenate([p[4] for p in ps]), vs)


def test_partition_covers_every_block_once():
    numels = [1000, 37 * 129, 4096, 5, 130 * 64, 1]
    for world in (1, 2, 3, 4, 8):
        seen = {}
        for r in range(world):
            for sh in sharding.partition(numels, world, r):
                assert sh.start % 128 == 0 and sh.numel > 0
                for e in range(sh.start, sh.start + sh.numel):
                    key = (sh.tensor, e)
                    assert key not in seen
                    seen[key] = r
        assert len(seen) == sum(numels)


def _clip_worker(rank, world, port, q):
    """Data-parallel global-norm clipping: each rank sums the squares of its
    own shards' gradients, one all-reduce (SUM) gives every rank the same
    total, and each rank steps its shards with the resulting factor."""
    from oracle import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.custom("mr", SHAPES, "zip_sr", flags=FLAGS)
        shards = sharding.partition([int(np.prod(s)) for s in SHAPES], world, rank)
        grads = [W.draw_grad(w, w.tensors[sh.tensor], sh.tensor, 1)[sh.start:sh.start + sh.numel].contiguous()
                 .view(torch.int16).numpy().view(np.uint16) for sh in shards]
        local = torch.tensor([float(O.grad_sqnorm(grads))], dtype=torch.float32)
        dist.all_reduce(local)
        clip = O.clip_factor(np.float32(local.item()), 0.05)
        h = W.HYPER
        outs = []
        for sh, g in zip(shards, grads):
            spec = w.tensors[sh.tensor]
            th = W.init_param(spec, sh.tensor).numpy()[sh.start:sh.start + sh.numel]
            t = O.OracleTensor.zeros_state(th, sh.tensor, flags=spec.flags, elem_offset=sh.elem_offset)
            t.step(g, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 1, 11, "zip_sr", 0, clip=clip)
            outs.append((sh.tensor, sh.start, t.param.copy()))
        gathered = [None] * world
        dist.all_gather_object(gathered, (float(local.item()), float(clip), outs))
        if rank == 0:
            q.put(gathered)
    finally:
        dist.destroy_process_group()


def test_two_rank_global_norm_clipping():
    from oracle import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_clip_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    totals = {g[0] for g in gathered}
    clips = {g[1] for g in gathered}
    assert len(totals) == 1 and len(clips) == 1            # every rank clips with the same factor
    total, clip = totals.pop(), clips.pop()
    # the all-reduced sum differs from the single-rank order only by rounding
    w = W.custom("mr", SHAPES, "zip_sr", flags=FLAGS)
    whole_g = [W.draw_grad(w, s, i, 1).view(torch.int16).numpy().view(np.uint16) for i, s in enumerate(w.tensors)]
    single = float(O.grad_sqnorm(whole_g))
    assert abs(total - single) <= 32 * 2.0 ** -24 * single
    assert clip < 1.0
    # with one factor the sharded step equals the whole-tensor step bit for bit
    h = W.HYPER
    parts = {}
    for _, _, outs in gathered:
        for tensor, start, th in outs:
            parts.setdefault(tensor, []).append((start, th))
    for i, s in enumerate(w.tensors):
        t = O.OracleTensor.zeros_state(W.init_param(s, i).numpy(), i, flags=s.flags)
        t.step(whole_g[i], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 1, 11, "zip_sr", 0,
               clip=np.float32(clip))
        ps = sorted(parts[i], key=lambda x: x[0])
        assert np.array_equal(np.concatenate([p[1] for p in ps]), t.param)


# ------------------------------------------------- factored statistics exchange
FSHAPES = [(48, 200), (300,), (64, 264), (33, 40)]
FFLAGS = [W.T_FACTORED, 0, W.T_FACTORED | W.T_LM_HEAD, W.T_FACTORED]


def _exact_grads(step):
    """Small integers times 2^-12 in BF16: float64 sums of their squares are
    exact in any order, so the sharded statistics equal the whole-tensor ones."""
    rng = np.random.default_rng(1000 + step)
    out = []
    for s in FSHAPES:
        x = rng.integers(-200, 201, int(np.prod(s))).astype(np.float32) * np.float32(2.0 ** -12)
        out.append(torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    return out


def _sums_floats_from_library(shards):
    """q4adamw_dp_sums_floats (host-only) for this rank's shard list."""
    import ctypes

    from bit_quantized_adamw_q4adamw_b300 import _native
    arr = (_native.Q4Tensor * len(shards))()
    fake = 1 << 40                       # never dereferenced by a host-only call
    full = (ctypes.c_int64 * len(shards))()
    for k, sh in enumerate(shards):
        s = FSHAPES[sh.tensor]
        d = arr[k]
        d.param = d.grad = d.m_codes = d.m_scale = d.v_codes = d.v_scale = d.v_row = d.v_col = fake
        d.numel, d.rows, d.elem_offset, d.flags = sh.numel, s[0] if len(s) == 2 else 1, sh.start, FFLAGS[sh.tensor]
        full[k] = int(np.prod(s))
    n = ctypes.c_int64()
    assert _native.lib().q4adamw_dp_sums_floats(arr, len(shards), 2, full, ctypes.byref(n)) == 0
    return n.value


def _factored_worker(rank, world, port, q):
    from oracle import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        numels = [int(np.prod(s)) for s in FSHAPES]
        shards = sharding.partition_all(numels, world, rank)
        h = W.HYPER
        ora = []
        for sh in shards:
            s = FSHAPES[sh.tensor]
            rows = s[0] if len(s) == 2 else 1
            fact = bool(FFLAGS[sh.tensor] & W.T_FACTORED)
            th = W.init_param(W.TensorSpec("p", s, FFLAGS[sh.tensor]), sh.tensor).numpy()[sh.start:sh.start + sh.numel]
            ora.append(O.OracleTensor.zeros_state(th, sh.tensor, rows=rows, flags=FFLAGS[sh.tensor],
                                                  elem_offset=sh.start, recipe="factored",
                                                  cols=numels[sh.tensor] // rows if fact else None))
        # the sums buffer: per factored tensor in list order, rows then columns
        # (the library's layout, whose size its host-only call states)
        layout = [(sh.tensor, o.rows, o.cols) for sh, o in zip(shards, ora) if o.factored]
        n_floats = sum(r + c for _, r, c in layout)
        assert _sums_floats_from_library(shards) == n_floats
        for step in (1, 2, 3):
            g = _exact_grads(step)
            buf = torch.zeros(n_floats, dtype=torch.float64)
            off = 0
            for sh, o in zip(shards, ora):
                if o.factored:
                    rs, cs = o.factored_partials(g[sh.tensor][sh.start:sh.start + sh.numel])
                    buf[off:off + o.rows] = torch.from_numpy(rs)
                    buf[off + o.rows:off + o.rows + o.cols] = torch.from_numpy(cs)
                    off += o.rows + o.cols
            dist.all_reduce(buf)                       # SUM over the data-parallel group
            off = 0
            for sh, o in zip(shards, ora):
                rs, cs = np.zeros(1), np.zeros(1)
                if o.factored:
                    rs = buf[off:off + o.rows].numpy()
                    cs = buf[off + o.rows:off + o.rows + o.cols].numpy()
                    off += o.rows + o.cols
                o.step_sums(g[sh.tensor][sh.start:sh.start + sh.numel], rs, cs, h["lr"], h["beta1"], h["beta2"],
                            h["eps"], h["weight_decay"], step, 5, "factored", O.LM_HEAD_SR_ACTIVE)
        outs = [(sh.tensor, sh.start, o.param.copy(), o.m_codes.copy(),
                 None if o.factored else o.v_codes.copy(),
                 o.v_row.copy() if o.factored else None, o.v_col.copy() if o.factored else None)
                for sh, o in zip(shards, ora)]
        gathered = [None] * world
        dist.all_gather_object(gathered, outs)
        if rank == 0:
            q.put(gathered)
    finally:
        dist.destroy_process_group()


def test_two_rank_factored_statistics_exchange():
    # AReno docs "State representation": under data parallelism each rank's
    # row and column sums are added over the group, and R and C are updated
    # from the totals.  Two
    # gloo ranks hold block-aligned shards (cut inside rows, one rank holding
    # no element of a parameter); after three steps every rank's R and C and
    # the union of the shards equal the single-rank step bit for bit.
    from oracle import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_factored_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    numels = [int(np.prod(s)) for s in FSHAPES]
    assert any(sh.numel == 0 for r in range(2) for sh in sharding.partition_all(numels, 2, r))
    h = W.HYPER
    for i, s in enumerate(FSHAPES):
        rows = s[0] if len(s) == 2 else 1
        t = O.OracleTensor.zeros_state(W.init_param(W.TensorSpec("p", s, FFLAGS[i]), i).numpy(), i, rows=rows,
                                       flags=FFLAGS[i], recipe="factored")
        for step in (1, 2, 3):
            t.step(_exact_grads(step)[i], h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], step, 5,
                   "factored", O.LM_HEAD_SR_ACTIVE)
        parts = sorted([o for outs in gathered for o in outs if o[0] == i and o[2].size > 0], key=lambda o: o[1])
        assert np.array_equal(np.concatenate([p[2] for p in parts]), t.param), i
        assert np.array_equal(np.concatenate([p[3] for p in parts]), t.m_codes), i
        if t.factored:
            for outs in gathered:                       # every rank's copy, the empty shard's too
                (o,) = [o for o in outs if o[0] == i]
                assert np.array_equal(o[5], t.v_row) and np.array_equal(o[6], t.v_col), i
        else:
            assert np.array_equal(np.concatenate([p[4] for p in parts]), t.v_codes), i
