"""Multi-process (gloo, world size 2) check of the data-parallel partition:
each rank evaluates only its units, the gathered parts equal the whole.
The per-rank evaluation is the CPU oracle, since these ranks have no GPU."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_27_gb300 import shard
from workloads import as_f64, make_inputs


def test_unit_ranges_cover_every_unit_once():
    for n in (1, 2, 5, 16, 17, 64):
        for world in (1, 2, 3, 4, 8):
            ranges = [shard.unit_range(r, world, n) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_unit_views_are_contiguous_slices():
    q = torch.arange(2 * 8 * 3 * 4).reshape(2, 8, 3, 4)
    v = shard.unit_view(q, 4, 1, 3)  # units of 4 heads: units 1..2
    assert v.is_contiguous() and v.shape == (2, 4, 3, 4)
    assert torch.equal(v[0], q[0, 4:8]) and torch.equal(v[1], q[1, 0:4])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, B, Hq, Hkv, N, d, causal, queue):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = make_inputs(B, Hq, Hkv, N, d, seed=21, with_grad=True)
    views, (Bs, Hqs, Hkvs) = shard.shard(inp, Hq, Hkv, rank, world)
    o, lse = oracle.attention_forward(as_f64(views["q"]), as_f64(views["k"]), as_f64(views["v"]),
                                      0.3, causal)
    dq, dk, dv = oracle.attention_backward(as_f64(views["q"]), as_f64(views["k"]),
                                           as_f64(views["v"]), as_f64(views["do"]), 0.3, causal)
    assert o.shape[:2] == (Bs, Hqs) and dk.shape[:2] == (Bs, Hkvs)
    parts = [None] * world
    dist.all_gather_object(parts, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})
    if rank == 0:
        full = {n: np.concatenate([p[n] for p in parts]) for n in parts[0]}
        queue.put({n: x for n, x in full.items()})
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("B,Hq,Hkv,causal", [(2, 4, 2, True), (1, 6, 3, False), (3, 2, 2, True)])
def test_two_ranks_reproduce_the_whole(B, Hq, Hkv, causal):
    import oracle
    N, d, world = 37, 8, 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, B, Hq, Hkv, N, d, causal, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inp = make_inputs(B, Hq, Hkv, N, d, seed=21, with_grad=True)
    f = {n: as_f64(t) for n, t in inp.items()}
    o, lse = oracle.attention_forward(f["q"], f["k"], f["v"], 0.3, causal)
    dq, dk, dv = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], 0.3, causal)
    G = Hq // Hkv
    # the gathered parts are unit-major views of the full tensors
    assert np.array_equal(got["o"], o.reshape(B * Hkv, G, N, d))
    assert np.array_equal(got["lse"], lse.reshape(B * Hkv, G, N))
    assert np.array_equal(got["dq"], dq.reshape(B * Hkv, G, N, d))
    assert np.array_equal(got["dk"], dk.reshape(B * Hkv, 1, N, d))
    assert np.array_equal(got["dv"], dv.reshape(B * Hkv, 1, N, d))
