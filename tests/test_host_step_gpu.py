"""muon_step_host: the step on parameters, gradients and momenta held in
host memory, streamed through a device staging buffer in units of whole
slices, copies overlapping the kernels.

It runs the same kernels on the same values as muon_step, so after each of
two steps the host parameters and momenta must equal, bit for bit, those of
muon_step on device copies of the same inputs.  Covered: units of the
minimum size (one slice per unit) and larger (several slices per unit, the
fused kernel's group in one unit), two to five buffers in rotation,
page-locked, pageable and muon_host_alloc (huge-page) host memory, and the
errors for a unit or a staging buffer too small, or a misaligned one.
"""
import pytest
import torch

from helpers import make_inputs, muon

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5)
SHAPES = [(3, 200, 150), (300, 200), (24, 10240), (2, 24, 10240), (130, 260)]


def _host_copies(m, ts, memory):
    """Host copies of ts: page-locked by torch, pageable, or views into one
    flat buffer from muon_host_alloc."""
    if memory == "pinned":
        return [t.clone().pin_memory() for t in ts]
    if memory == "pageable":
        return [t.clone() for t in ts]
    buf = m.alloc_host(sum(t.numel() for t in ts), ts[0].dtype)
    out, off = [], 0
    for t in ts:
        v = buf[off:off + t.numel()].view(t.shape)
        v.copy_(t)
        out.append(v)
        off += t.numel()
    return out


@pytest.mark.parametrize("units", [(1, 3), (4, 2), (2, 5)], ids=["min-x3", "4x-x2", "2x-x5"])
@pytest.mark.parametrize("memory", ["pinned", "pageable", "huge"])
def test_host_step_equals_device_step_twice(units, memory):
    m = muon()
    W, Gs, M = make_inputs(SHAPES, torch.bfloat16, steps=2)
    plan = m.Plan([(s, torch.bfloat16) for s in SHAPES])
    # device reference
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    ws_d = m.alloc_workspace(plan)
    # host state
    Wh = _host_copies(m, W, memory)
    Mh = _host_copies(m, M, memory)
    ws = m.alloc_workspace(plan)
    unit = plan.host_unit_bytes * units[0]
    staging = torch.empty(unit * units[1], dtype=torch.uint8, device="cuda")
    for t in range(2):
        Gh = _host_copies(m, Gs[t], memory)
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


def test_alloc_host_memory_is_zeroed_aligned_on_huge_pages_and_freed():
    import ctypes
    import gc
    m = muon()
    x = m.alloc_host(3 << 20, torch.float32)          # 12 MiB
    assert x.numel() == 3 << 20 and not x.is_cuda and bool((x == 0).all())
    addr = x.data_ptr()
    hp = int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
    assert addr % hp == 0
    thp = open("/sys/kernel/mm/transparent_hugepage/enabled").read()
    if "[never]" not in thp:
        # the mapping holding the buffer is backed by transparent huge pages
        huge, inside = None, False
        for line in open("/proc/self/smaps"):
            f = line.split()
            if "-" in f[0] and ":" not in f[0]:
                lo, hi = (int(v, 16) for v in f[0].split("-"))
                inside = lo <= addr < hi
            elif inside and f[0] == "AnonHugePages:":
                huge = int(f[1])
        assert huge is not None and huge > 0, huge
    # the device reads and writes it (the copy engines, page-locked)
    d = torch.arange(x.numel(), dtype=torch.float32, device="cuda")
    x.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(x[:1000], torch.arange(1000, dtype=torch.float32))
    view = x[5:10]
    del x, d
    gc.collect()
    assert view[0].item() == 5.0                       # a view keeps the memory
    del view
    gc.collect()
    # the last view is gone: the memory was handed back, so the address is
    # unknown to muon_host_free now
    assert m.load().muon_host_free(ctypes.c_void_p(addr)) == -1
