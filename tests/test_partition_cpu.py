"""The replica path on the CPU: gloo ranks that each hold every parameter
and the full gradients update only the slices muon_plan_partition gives them
(here with the fp64 oracle standing in for the GPU update, rounded to the
parameter dtype), then Partition.broadcast sends every slice from its owner.
Every rank must end with the parameters of the single-replica oracle step,
bit for bit, and hold momentum only for its own slices."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

SHAPES = [((3, 24, 200), torch.bfloat16), ((40, 24), torch.bfloat16), ((2, 30, 50), torch.float32),
          ((24, 200), torch.bfloat16), ((50, 30), torch.float32), ((4, 16, 64), torch.bfloat16)]
HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    import synth
    W = [synth.draw(s, 0.02, synth.param_seed(1, i), dt) for i, (s, dt) in enumerate(SHAPES)]
    G = [synth.draw(s, 1e-2, synth.param_seed(0, i), dt) for i, (s, dt) in enumerate(SHAPES)]
    return W, G


def _oracle_update(w, g, mom):
    """fp64 oracle step of one 2-D slice, W' rounded to the slice's dtype."""
    import oracle
    wo, mo, _ = oracle.muon_slice(w, g, mom, HP["lr"], HP["beta"], HP["wd"], HP["nesterov"])
    return torch.from_numpy(wo).to(w.dtype), torch.from_numpy(mo).float()


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import newton_schulz_05_gb300 as m
    dist.init_process_group("gloo", rank=rank, world_size=world)
    W, G = _inputs()
    plan = m.Plan([w for w in W])
    part = m.Partition(plan, world)
    # this rank's update of its own slices, momentum only for them
    mine = part.owned(rank)
    moms = []
    for (p, e), wv, gv in zip(mine, part.views(W, rank), part.views(G, rank)):
        w1, m1 = _oracle_update(wv, gv, torch.zeros(wv.shape))
        wv.copy_(w1)
        moms.append(m1)
    part.broadcast(W)
    out[rank] = ([w.clone() for w in W], mine, moms)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replicas_update_their_slices_and_broadcast(world):
    from newton_schulz_05_gb300 import build
    build.build()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    W, G = _inputs()
    expect = []
    for w, g in zip(W, G):
        ws = [w] if w.dim() == 2 else list(w)
        gs = [g] if g.dim() == 2 else list(g)
        res = [_oracle_update(a, b, torch.zeros(a.shape)) for a, b in zip(ws, gs)]
        expect.append((torch.stack([r[0] for r in res]).reshape(w.shape),
                       torch.stack([r[1] for r in res]).reshape(w.shape)))
    seen = set()
    for r in range(world):
        params, mine, moms = out[r]
        for p, (e_w, _) in enumerate(expect):
            assert torch.equal(params[p], e_w), (r, p)
        for (p, e), mom in zip(mine, moms):
            assert (p, e) not in seen
            seen.add((p, e))
            ref = expect[p][1] if expect[p][1].dim() == 2 else expect[p][1][e]
            assert torch.equal(mom, ref)
    # every slice was updated by exactly one rank
    assert len(seen) == sum(s[0] if len(s) == 3 else 1 for s, _ in SHAPES)
