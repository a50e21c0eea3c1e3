"""Gradient reduction overlapped with backward (GradReduceOverlap), on gloo
ranks on the CPU: the data-parallel step that feeds the Muon optimizer
(Paddle PR "Support Muon sharding optimizer comm overlap": backward hooks
fill reduction buffers, matrix and other parameters in separate buffers,
shared weights in a buffer reduced after backward, and the loss scaler
checks only fully reduced gradients).

Every rank holds the same model and a different batch.  The reduced
gradients must equal the mean over ranks of the gradients a plain backward
gives: bit for bit with two ranks (a + b is the same number in either
order), to fp32 rounding with three.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


class _Net(torch.nn.Module):
    """Embedding, two linear layers and a layer norm, with the output
    projection tied to the embedding (a shared weight)."""

    def __init__(self):
        super().__init__()
        g = torch.Generator().manual_seed(7)
        self.emb = torch.nn.Embedding(50, 16)
        self.lin1 = torch.nn.Linear(16, 32)
        self.ln = torch.nn.LayerNorm(32)
        self.lin2 = torch.nn.Linear(32, 16)
        with torch.no_grad():
            for p in self.parameters():
                p.copy_(torch.randn(p.shape, generator=g) * 0.1)

    def forward(self, x):
        h = self.emb(x)
        h = self.ln(torch.relu(self.lin1(h)))
        h = self.lin2(h)
        return h @ self.emb.weight.t()


def _loss(net, rank, micro=0):
    g = torch.Generator().manual_seed(1000 * rank + micro)
    x = torch.randint(0, 50, (4, 6), generator=g)
    y = torch.randint(0, 50, (4, 6), generator=g)
    return torch.nn.functional.cross_entropy(net(x).reshape(-1, 50), y.reshape(-1))


def _reference(world, rank, micro_batches):
    """Mean over ranks of plain-backward gradients (all ranks' local
    gradients gathered, summed in rank order)."""
    net = _Net()
    for mb in range(micro_batches):
        _loss(net, rank, mb).backward()
    out = []
    for p in net.parameters():
        parts = [torch.empty_like(p.grad) for _ in range(world)]
        dist.all_gather(parts, p.grad.contiguous())
        s = parts[0].clone()
        for q in parts[1:]:
            s += q
        out.append(s / world)
    return out


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from newton_schulz_05_gb300.comm import GradReduceOverlap
    res = {}
    for case in ("hooks", "tied_sync_only", "micro_batches"):
        net = _Net()
        params = list(net.parameters())
        sync = [net.emb.weight] if case == "tied_sync_only" else []
        ov = GradReduceOverlap(params, bucket_bytes=1024, sync_only=sync)
        kinds = {b.kind for b in ov.buckets}
        mbs = 2 if case == "micro_batches" else 1
        for mb in range(mbs):
            ov.begin(last_micro_batch=(mb == mbs - 1))
            _loss(net, rank, mb).backward()
        grads = ov.finish()
        ref = _reference(world, rank, mbs)
        if world == 2:
            same = all(torch.equal(a, b) for a, b in zip(grads, ref))
        else:
            same = all(torch.allclose(a, b, rtol=1e-6, atol=1e-8) for a, b in zip(grads, ref))
        res[case] = (same, ov.overlapped_buckets(), len(ov.buckets), sorted(kinds),
                     all(p.grad is None for p in params))
        ov.remove()
    # a non-finite gradient on one rank reaches every rank through the
    # reduction, so a loss scaler that checks after finish() skips everywhere
    net = _Net()
    ov = GradReduceOverlap(list(net.parameters()), bucket_bytes=1024)
    if rank == world - 1:
        net.lin1.weight.register_hook(lambda g: g.index_fill(0, torch.tensor([0]), float("inf")))
    ov.begin()
    _loss(net, rank).backward()
    grads = ov.finish()
    res["found_inf"] = not all(torch.isfinite(g).all() for g in grads)
    # hooks fire only between begin() and finish()
    net = _Net()
    ov = GradReduceOverlap(list(net.parameters()))
    try:
        _loss(net, rank).backward()
        res["unarmed"] = "no error"
    except RuntimeError as e:
        res["unarmed"] = str(e)
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_overlapped_reduction_equals_reduce_after_backward(world):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        res = out[r]
        for case in ("hooks", "tied_sync_only", "micro_batches"):
            same, early, nb, kinds, freed = res[case]
            assert same, (r, case)
            # matrix and other parameters in separate buffers, several buffers,
            # at least one reduction started while backward was still running
            assert kinds == ["matrix", "other"] and nb >= 3 and early >= 1, (r, case, nb, early)
            assert freed, (r, case)
        assert res["found_inf"], r
        assert "begin() was not called" in res["unarmed"], res["unarmed"]


def test_single_process_reduction_is_the_plain_gradient():
    from newton_schulz_05_gb300.comm import GradReduceOverlap
    net = _Net()
    ref = _Net()
    _loss(ref, 0).backward()
    ov = GradReduceOverlap(list(net.parameters()), bucket_bytes=1024)
    ov.begin()
    _loss(net, 0).backward()
    grads = ov.finish()
    assert all(torch.equal(a, b.grad) for a, b in zip(grads, ref.parameters()))
