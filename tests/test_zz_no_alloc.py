"""muon_step_static: the Muon step for callers that cannot allocate device
memory (a runtime whose own pooled allocator holds nearly all of the GPU's
memory, or a latency-bound caller that cannot afford a blocking cudaMalloc).
Its scratch is a static device array inside the library.

Through the C ABI, two steps in a row with muon_step_static must match two
steps of muon_step with a caller-allocated workspace, within the tolerances
of the other parity tests: momentum within 1e-6 relative, bf16 parameters
within one bf16 ulp.  Plans that need more scratch than the static array
holds are rejected before any device work.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bf16_ulp, make_inputs, muon

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


def test_static_scratch_step_matches_workspace_step_twice():
    m = muon()
    L = m.load()
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
        torch.cuda.synchronize()
        for wa, wb, ma, mb in zip(Wa, Wb, Ma, Mb):
            a = wa.double().cpu().numpy(); b = wb.double().cpu().numpy()
            assert np.all(np.abs(a - b) <= bf16_ulp(a)), "step %d: parameters differ" % t
            x = ma.double().cpu().numpy(); y = mb.double().cpu().numpy()
            assert np.all(np.abs(x - y) <= 1e-6 * np.abs(x) + 1e-30), "step %d: momentum differs" % t


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
