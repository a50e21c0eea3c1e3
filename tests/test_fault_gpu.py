"""Bounded device waits driven to expiry, without any GPU fault.

MUON_FAULT=timeout gives every bounded wait of the step kernels a budget of
zero polls, so the first wait of each kernel gives up at once.  The step must
then report MUON_ERR_DEVICE_TIMEOUT through the workspace error word (or,
for the static-scratch step, through muon_static_error), leave every
parameter as it was, and leave the stream, the context and the workspace
usable: after the word is cleared, the next step runs normally and gives the
same bits as the same step on a fresh workspace.  The kernels still wait,
with the normal budget, for the copies they already issued, so nothing is in
flight when they return.
"""
import pytest
import torch

from helpers import make_inputs, muon

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5)
TIMEOUT = -6


@pytest.mark.parametrize("shapes", [[(24, 10240)] * 4, [(2, 200, 150), (300, 200)]],
                         ids=["skinny", "dense"])
def test_timeout_is_reported_and_the_next_step_runs(shapes, monkeypatch):
    m = muon()
    W, Gs, M = make_inputs(shapes, torch.bfloat16, steps=2)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    skinny = plan.groups()[0]["kernel"] == m.KERNEL_SKINNY
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    ws = m.alloc_workspace(plan)
    G0 = [g.cuda() for g in Gs[0]]
    monkeypatch.setenv("MUON_FAULT", "timeout")
    m.step(plan, Wd, G0, Md, workspace=ws, **HP)
    torch.cuda.synchronize()
    monkeypatch.delenv("MUON_FAULT")
    assert m.workspace_error(ws, clear=True) == TIMEOUT
    assert all(torch.equal(a.cpu(), b) for a, b in zip(Wd, W)), "parameters changed"
    if skinny:
        # the fused kernel stores no momentum once its first wait gave up
        assert all(torch.equal(a.cpu(), b) for a, b in zip(Md, M)), "momentum changed"
    # the word is clear; the next step on the same workspace runs normally
    assert m.workspace_error(ws) == 0
    Wr = [x.clone() for x in Wd]; Mr = [x.clone() for x in Md]
    G1 = [g.cuda() for g in Gs[1]]
    m.step(plan, Wd, G1, Md, workspace=ws, **HP)
    torch.cuda.synchronize()
    assert m.workspace_error(ws) == 0
    ws2 = m.alloc_workspace(plan)
    m.step(plan, Wr, G1, Mr, workspace=ws2, **HP)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(Wd, Wr))
    assert all(torch.equal(a, b) for a, b in zip(Md, Mr))
    assert any(not torch.equal(a.cpu(), b) for a, b in zip(Wd, W))


def test_static_scratch_step_reports_timeout(monkeypatch):
    m = muon()
    shapes = [(2, 200, 150), (24, 700)]
    W, Gs, M = make_inputs(shapes, torch.bfloat16)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    G = [g.cuda() for g in Gs[0]]
    monkeypatch.setenv("MUON_FAULT", "timeout")
    m.step_static(plan, Wd, G, Md, **HP)
    torch.cuda.synchronize()
    monkeypatch.delenv("MUON_FAULT")
    assert m.static_error(clear=True) == TIMEOUT
    assert all(torch.equal(a.cpu(), b) for a, b in zip(Wd, W))
    m.step_static(plan, Wd, G, Md, **HP)
    assert m.static_error() == 0
