"""muon_step_host: the step on parameters, gradients and momenta held in
host memory, streamed through a device staging buffer in units of whole
slices, copies overlapping the kernels.

It runs the same kernels on the same values as muon_step, so after each of
two steps the host parameters and momenta must equal, bit for bit, those of
muon_step on device copies of the same inputs.  Covered: units of the
minimum size (one slice per unit) and larger (several slices per unit, the
fused kernel's group in one unit), two to five buffers in rotation,
page-locked and pageable host memory, and the errors for a unit or a
staging buffer too small, or a misaligned one.
"""
import pytest
import torch

from helpers import make_inputs, muon

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5)
SHAPES = [(3, 200, 150), (300, 200), (24, 10240), (2, 24, 10240), (130, 260)]


@pytest.mark.parametrize("units", [(1, 3), (4, 2), (2, 5)], ids=["min-x3", "4x-x2", "2x-x5"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_step_equals_device_step_twice(units, pinned):
    m = muon()
    W, Gs, M = make_inputs(SHAPES, torch.bfloat16, steps=2)
    plan = m.Plan([(s, torch.bfloat16) for s in SHAPES])
    # device reference
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    ws_d = m.alloc_workspace(plan)
    # host state
    Wh = [w.clone().pin_memory() if pinned else w.clone() for w in W]
    Mh = [x.clone().pin_memory() if pinned else x.clone() for x in M]
    ws = m.alloc_workspace(plan)
    unit = plan.host_unit_bytes * units[0]
    staging = torch.empty(unit * units[1], dtype=torch.uint8, device="cuda")
    for t in range(2):
        Gh = [g.clone().pin_memory() if pinned else g.clone() for g in Gs[t]]
        m.step(plan, Wd, [g.cuda() for g in Gs[t]], Md, workspace=ws_d, **HP)
        m.PreparedHostStep(plan, Wh, Gh, Mh, workspace=ws, staging=staging, unit_bytes=unit,
                           **HP)()
        torch.cuda.synchronize()
        assert m.workspace_error(ws) == 0 and m.workspace_error(ws_d) == 0
        for a, b in zip(Wh, Wd):
            assert torch.equal(a, b.cpu()), "step %d: parameters differ" % t
        for a, b in zip(Mh, Md):
            assert torch.equal(a, b.cpu()), "step %d: momentum differs" % t


def test_host_step_rejects_small_or_misaligned_staging():
    m = muon()
    L = m.load()
    import ctypes
    plan = m.Plan([(s, torch.bfloat16) for s in SHAPES])
    W, Gs, M = make_inputs(SHAPES, torch.bfloat16)
    ws = m.alloc_workspace(plan)
    unit = plan.host_unit_bytes
    small = torch.empty(3 * unit, dtype=torch.uint8, device="cuda")
    for u, buf in ((unit - 256, small), (unit, small[:unit + 256])):
        # a slice larger than a unit, or room for fewer than two units
        with pytest.raises(m.MuonError) as e:
            m.PreparedHostStep(plan, W, Gs[0], M, workspace=ws, staging=buf, unit_bytes=u, **HP)()
        assert e.value.status == -7
    big = torch.empty(3 * unit + 512, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p * len(W)
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    rc = L.muon_step_host(plan.handle, P(*[x.data_ptr() for x in W]),
                          P(*[x.data_ptr() for x in Gs[0]]), P(*[x.data_ptr() for x in M]),
                          0.02, 0.95, 0.1, 1, 5, c, ctypes.c_void_p(ws.data_ptr()),
                          ws.numel(), ctypes.c_void_p(big.data_ptr() + 16), 3 * unit, unit,
                          None)
    assert rc == -4
