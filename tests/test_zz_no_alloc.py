"""muon_step_static: the Muon step for callers that cannot allocate device
memory (a runtime whose own pooled allocator holds nearly all of the GPU's
memory, or a latency-bound caller that cannot afford a blocking cudaMalloc).
Its scratch is a static device array inside the library.

Through the C ABI, two steps in a row with muon_step_static must give the
same bits as two steps of muon_step with a caller-allocated workspace: both
run the same plan, chunking and deterministic kernels on the same inputs.
Before the compared steps the static array is filled by a step of another
plan, so a value read before it is written would show.  After each step the
static array's error word reads zero.  Plans that need more scratch than the
static array holds are rejected before any device work.  This file is
collected last.
"""
import ctypes

import pytest
import torch

from helpers import make_inputs, muon

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5)
COEFFS = (3.4445, -4.7750, 2.0315)


def _c_step(L, plan, W, G, M, static, ws=None):
    P = ctypes.c_void_p * len(W)
    pw = P(*[x.data_ptr() for x in W]); pg = P(*[x.data_ptr() for x in G])
    pm = P(*[x.data_ptr() for x in M])
    c = (ctypes.c_float * 3)(*COEFFS)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [plan.handle, pw, pg, pm, HP["lr"], HP["beta"], HP["wd"], 1, HP["ns_steps"], c]
    if static:
        return L.muon_step_static(*args, stream)
    return L.muon_step(*args, ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)


def _static_error(L):
    code = ctypes.c_int(-99)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.muon_static_error(stream, 1, ctypes.byref(code)) == 0
    return code.value


def test_static_scratch_step_matches_workspace_step_twice():
    m = muon()
    L = m.load()
    # fill the static array with another plan's scratch first
    other = [(3, 256, 384)]
    Wo, Go, Mo = make_inputs(other, torch.bfloat16)
    po = m.Plan([(s, torch.bfloat16) for s in other])
    assert 256 < po.workspace_bytes <= m.STATIC_WORKSPACE_BYTES
    assert _c_step(L, po, [Wo[0].cuda()], [Go[0][0].cuda()], [Mo[0].cuda()], static=True) == 0
    assert _static_error(L) == 0
    # dense groups (their scratch is the static array) plus a skinny group
    shapes = [(2, 200, 150), (300, 200), (24, 700)]
    W, Gs, M = make_inputs(shapes, torch.bfloat16, steps=2)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    assert 256 < plan.workspace_bytes <= m.STATIC_WORKSPACE_BYTES
    Wa = [w.cuda() for w in W]; Ma = [x.cuda() for x in M]
    Wb = [w.cuda() for w in W]; Mb = [x.cuda() for x in M]
    ws = m.alloc_workspace(plan)
    for t in range(2):
        G = [g.cuda() for g in Gs[t]]
        assert _c_step(L, plan, Wa, G, Ma, static=False, ws=ws) == 0
        assert _c_step(L, plan, Wb, G, Mb, static=True) == 0
        assert _static_error(L) == 0
        torch.cuda.synchronize()
        assert m.workspace_error(ws) == 0
        for wa, wb, ma, mb in zip(Wa, Wb, Ma, Mb):
            assert torch.equal(wa, wb), "step %d: parameters differ" % t
            assert torch.equal(ma, mb), "step %d: momentum differs" % t


def test_static_scratch_rejects_plans_that_do_not_fit():
    m = muon()
    L = m.load()
    plan = m.Plan([((4096, 4096), torch.bfloat16)])
    assert plan.workspace_bytes > m.STATIC_WORKSPACE_BYTES
    P = ctypes.c_void_p * 1
    dummy = P(ctypes.c_void_p(0x1000))
    c = (ctypes.c_float * 3)(*COEFFS)
    rc = L.muon_step_static(plan.handle, dummy, dummy, dummy, 0.02, 0.95, 0.1, 1, 5, c, None)
    assert rc == -7 and m.status_string(rc) == "workspace too small for the plan"
