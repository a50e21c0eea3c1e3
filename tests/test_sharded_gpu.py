"""The replica path on one GPU: the ranks of a ShardedMuon group run one
after another on the same parameter tensors (each writes only its own
slices, so no broadcast is needed to assemble the result).  Every slice is
computed independently of the others, so the assembled parameters and the
ranks' momentum must equal the single-replica Muon step bit for bit, for
skinny, dense, transposed and expert-stack slices."""
import pytest
import torch

import synth
from helpers import muon

pytestmark = pytest.mark.gpu

SHAPES = [(4, 24, 1024), (24, 10240), (2, 200, 300), (300, 200), (3, 64, 512), (130, 130),
          (10240, 24)]


def _inputs(steps):
    W = [synth.draw(s, 0.02, synth.param_seed(1, i), torch.bfloat16, "cuda") for i, s in enumerate(SHAPES)]
    Gs = [[synth.draw(s, 1e-2, synth.param_seed(t, i), torch.bfloat16, "cuda")
           for i, s in enumerate(SHAPES)] for t in range(steps)]
    return W, Gs


@pytest.mark.parametrize("world", [2, 3, 8])
def test_ranks_in_turn_equal_the_single_replica_step(world):
    m = muon()
    steps = 3
    W_ref, Gs = _inputs(steps)
    W = [w.clone() for w in W_ref]
    ref = m.Muon(W_ref)
    ranks = [m.ShardedMuon(W, r, world) for r in range(world)]
    for t in range(steps):
        ref.step(Gs[t])
        for sh in ranks:
            sh.update_owned(Gs[t])
        torch.cuda.synchronize()
        for p in range(len(SHAPES)):
            assert torch.equal(W[p], W_ref[p]), (t, p)
        for sh in ranks:
            assert m.workspace_error(sh.workspace) == 0
            for (p, e), mom in zip(sh.owned, sh.momentum):
                full = ref.momentum[p] if ref.momentum[p].dim() == 2 else ref.momentum[p][e]
                assert torch.equal(mom, full), (t, p, e)
    owned = [k for sh in ranks for k in sh.owned]
    assert len(owned) == len(set(owned)) == sum(s[0] if len(s) == 3 else 1 for s in SHAPES)


def test_one_replica_is_the_plain_step():
    m = muon()
    W_ref, Gs = _inputs(1)
    W = [w.clone() for w in W_ref]
    m.Muon(W_ref).step(Gs[0])
    m.ShardedMuon(W, 0, 1).step(Gs[0])
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(W, W_ref))
