"""The C-ABI boundary on the CPU: the library loads, exports every symbol the
header declares, and its host-only planner equals the oracle's plan bit for
bit (group ids, indices, dims, transposition flag, float bits of the scale).
No compute call is made here; muon_plan touches no device."""
import ctypes
import os
import re
import struct

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def muon():
    from newton_schulz_05_gb300 import build
    build.build()
    import newton_schulz_05_gb300 as m
    m.load()
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "muon.h")).read()
    return sorted(set(re.findall(r"MUON_API\s+[\w\s\*]+?\b(muon_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for f in ["muon_plan", "muon_step", "muon_plan_destroy", "muon_status_string"]:
        assert f in fns


def test_library_exports_every_declared_symbol(muon):
    L = muon.load()
    for f in header_functions():
        assert hasattr(L, f), f
    assert sorted(header_functions()) == sorted(muon.EXPORTS)


def _oracle_dt(d):
    return "bf16" if d == 0 else "f32"


def _compare_plan(muon, shapes, dtypes_t, **kw):
    import torch
    plan = muon.Plan([(s, d) for s, d in zip(shapes, dtypes_t)], **kw)
    dts = ["bf16" if d == torch.bfloat16 else "f32" for d in dtypes_t]
    sg, si, groups = oracle.plan(shapes, dts, scale_mode=kw.get("scale_mode", "sqrt_ratio"))
    got = plan.groups()
    assert len(got) == len(groups)
    for a, b in zip(got, groups):
        assert (a["M"], a["N"], a["count"], bool(a["tr"])) == (b["M"], b["N"], b["count"], b["tr"])
        assert _oracle_dt(a["dtype"]) == b["dtype"]
        assert struct.pack("<f", a["scale"]) == struct.pack("<f", b["scale"])
        assert (a["m"], a["n"]) == (min(a["M"], a["N"]), max(a["M"], a["N"]))
    s = 0
    for p, shp in enumerate(shapes):
        E = shp[0] if len(shp) == 3 else 1
        for e in range(E):
            assert plan.slice(p, e) == (sg[s], si[s])
            s += 1
    assert plan.num_slices == s
    return plan


def test_plan_matches_oracle_random(muon):
    import torch
    rng = np.random.default_rng(21)
    dims = [1, 7, 24, 64, 65, 130, 1408]
    for _ in range(40):
        shapes, dts = [], []
        for _ in range(rng.integers(1, 10)):
            if rng.random() < 0.4:
                shapes.append((int(rng.integers(1, 4)), int(rng.choice(dims)), int(rng.choice(dims))))
            else:
                shapes.append((int(rng.choice(dims)), int(rng.choice(dims))))
            dts.append(torch.bfloat16 if rng.random() < 0.7 else torch.float32)
        _compare_plan(muon, shapes, dts)
        _compare_plan(muon, shapes, dts, mode="fp32")
        _compare_plan(muon, shapes, dts, scale_mode="rms_match")


def test_plan_log_lines(muon):
    # MUON_LOG=1: muon_plan prints one line per group to stderr
    import subprocess
    import sys
    code = ("import torch, newton_schulz_05_gb300 as m; "
            "m.Plan([((24, 10240), torch.bfloat16), ((2, 1408, 2048), torch.bfloat16), "
            "((2048, 1408), torch.bfloat16)])")
    env = dict(os.environ, MUON_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stderr.splitlines() if x.startswith("muon_plan:")]
    assert lines[0].startswith("muon_plan: 3 parameters, 4 slices, 3 groups, workspace ")
    assert "group 0 [24,10240] bf16 slices=1 m=24 n=10240 tr=0 scale=1 kernel=skinny cluster=2" \
        in lines[1]
    assert "group 1 [1408,2048] bf16 slices=2 m=1408 n=2048 tr=0" in lines[2] and \
        "kernel=dense chunk=2" in lines[2]
    assert "group 2 [2048,1408] bf16 slices=1 m=1408 n=2048 tr=1 scale=1.20604539" in lines[3]
    env.pop("MUON_LOG")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert "muon_plan:" not in r.stderr


def test_fault_switches_return_status_codes(muon, monkeypatch):
    # MUON_FAULT=alloc: the plan fails as if host memory ran out; =launch:
    # the step reports a failed launch after validating its arguments
    import torch
    monkeypatch.setenv("MUON_FAULT", "alloc")
    with pytest.raises(muon.MuonError) as e:
        muon.Plan([((24, 1000), torch.bfloat16)])
    assert e.value.status == -8
    monkeypatch.setenv("MUON_FAULT", "launch")
    plan = muon.Plan([((24, 1000), torch.bfloat16)])
    L = muon.load()
    P = ctypes.c_void_p * 1
    fake = P(ctypes.c_void_p(0x10000))
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    rc = L.muon_step(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c,
                     ctypes.c_void_p(0x100000), plan.workspace_bytes, None)
    assert rc == -5
    rc = L.muon_step(plan.handle, fake, fake, fake, float("nan"), 0.95, 0.1, 1, 5, c,
                     ctypes.c_void_p(0x100000), plan.workspace_bytes, None)
    assert rc == -1   # argument checks still come first
    monkeypatch.delenv("MUON_FAULT")


@pytest.mark.parametrize("name", ["fp32_24x1024", "skinny_74x24x10240", "stacks_experts",
                                  "dense_24L", "moe_24L"])
def test_plan_matches_oracle_on_workloads(muon, name):
    import synth
    w = synth.workload(name)
    plan = _compare_plan(muon, list(w.shapes), [w.dtype] * len(w.shapes))
    kinds = {(g["m"], g["n"]): g["kernel"] for g in plan.groups()}
    # the [24, 10240] batches run fused on chip, the rest on the dense path
    for (m, n), k in kinds.items():
        assert k == (muon.KERNEL_SKINNY if m <= 64 else muon.KERNEL_DENSE)


def test_plan_skinny_cluster_configuration(muon):
    import torch
    plan = muon.Plan([((24, 10240), torch.bfloat16)] * 74)
    (g,) = plan.groups()
    assert g["kernel"] == muon.KERNEL_SKINNY and g["cluster"] == 2 and g["count"] == 74
    assert plan.launches(5) == 1
    assert plan.workspace_bytes == 256


def test_plan_rejects_bad_input(muon):
    import torch
    with pytest.raises(muon.MuonError) as e:
        muon.Plan([((5,), torch.bfloat16)])
    assert e.value.status == -2
    with pytest.raises(muon.MuonError) as e:
        muon.Plan([((0, 4), torch.bfloat16)])
    assert e.value.status == -2
    with pytest.raises(muon.MuonError) as e:
        muon.Plan([((3, 4), 7)])
    assert e.value.status == -3
    L = muon.load()
    assert L.muon_plan(None, 1, None, None) == -1
    assert muon.status_string(-7) == "workspace too small for the plan"


def test_step_rejects_bad_arguments_before_any_launch(muon):
    # argument checks run on the host and return before touching a device
    import torch
    plan = muon.Plan([((24, 64), torch.bfloat16)])
    L = muon.load()
    P = ctypes.c_void_p * 1
    fake = P(ctypes.c_void_p(0x1000))
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    # null workspace
    assert L.muon_step(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c, None, 256, None) == -1
    # misaligned workspace
    assert L.muon_step(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c,
                       ctypes.c_void_p(0x1008), 4096, None) == -4
    # workspace too small
    assert L.muon_step(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c,
                       ctypes.c_void_p(0x1000), 16, None) == -7
    # negative step count, null parameter pointer, non-finite lr
    assert L.muon_step(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, -1, c,
                       ctypes.c_void_p(0x1000), 4096, None) == -1
    nul = P(ctypes.c_void_p(0))
    assert L.muon_step(plan.handle, nul, fake, fake, 0.02, 0.95, 0.1, 1, 5, c,
                       ctypes.c_void_p(0x1000), 4096, None) == -1
    assert L.muon_step(plan.handle, fake, fake, fake, float("nan"), 0.95, 0.1, 1, 5, c,
                       ctypes.c_void_p(0x1000), 4096, None) == -1
    assert L.muon_step_ortho(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c,
                             ctypes.c_void_p(0x1000), 4096, None, None) == -1


def test_workspace_cap_chunks_dense_groups(muon):
    import torch
    shapes = [((4, 300, 200), torch.bfloat16)]
    full = muon.Plan(shapes)
    (g,) = full.groups()
    assert g["kernel"] == muon.KERNEL_DENSE and g["chunk"] == 4
    # header, chunk x slice workspace, then one exponent slot per dense slice
    # (4 slots, padded to 256 bytes)
    exp_region = 256
    per = (full.workspace_bytes - 256 - exp_region) // 4
    capped = muon.Plan(shapes, workspace_cap=256 + 2 * per + exp_region)
    assert capped.groups()[0]["chunk"] == 2
    assert capped.workspace_bytes == 256 + 2 * per + exp_region
    assert capped.launches(5) == 2 * full.launches(5)


def test_amp_step_rejects_bad_arguments(muon):
    import torch
    plan = muon.Plan([((24, 64), torch.bfloat16)])
    L = muon.load()
    P = ctypes.c_void_p * 1
    fake = P(ctypes.c_void_p(0x1000))
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    # null found_inf, non-finite inv_scale
    assert L.muon_step_amp(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c, 1.0, None,
                           ctypes.c_void_p(0x1000), 4096, None) == -1
    assert L.muon_step_amp(plan.handle, fake, fake, fake, 0.02, 0.95, 0.1, 1, 5, c, float("inf"),
                           ctypes.c_void_p(0x2000), ctypes.c_void_p(0x1000), 4096, None) == -1


def test_adamw_rejects_bad_arguments(muon):
    L = muon.load()
    P = ctypes.c_void_p * 1
    fake = P(ctypes.c_void_p(0x1000))
    n = (ctypes.c_int64 * 1)(10)
    args = lambda **kw: [kw.get("n", 1), fake, fake, fake, fake, n, kw.get("dt", 0), 1e-3,
                         kw.get("b1", 0.9), 0.999, 1e-8, 0.0, kw.get("t", 1), None]
    assert L.muon_adamw_step(*args(t=0)) == -1
    assert L.muon_adamw_step(*args(b1=1.0)) == -1
    assert L.muon_adamw_step(*args(dt=5)) == -3
    assert L.muon_adamw_step(*args(n=-1)) == -1
    assert L.muon_adamw_step(0, None, None, None, None, None, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None) == 0


def _oracle_partition(plan, world, T, fr, br):
    dts = ["bf16" if d == 0 else "f32" for d in plan.dtypes]
    return oracle.partition(oracle.slice_costs(plan.shapes, dts, T, fr, br), world)


def test_partition_matches_oracle_random(muon):
    import torch
    rng = np.random.default_rng(5)
    dims = [1, 7, 24, 64, 65, 130, 1408, 4096]
    for _ in range(40):
        shapes = []
        for _ in range(rng.integers(1, 12)):
            if rng.random() < 0.4:
                shapes.append(((int(rng.integers(1, 6)), int(rng.choice(dims)), int(rng.choice(dims))),
                               torch.bfloat16 if rng.random() < 0.7 else torch.float32))
            else:
                shapes.append(((int(rng.choice(dims)), int(rng.choice(dims))),
                               torch.bfloat16 if rng.random() < 0.7 else torch.float32))
        plan = muon.Plan(shapes)
        world = int(rng.integers(1, 9))
        T = int(rng.integers(0, 8))
        fr, br = float(rng.choice([1.88e15, 1e9, 1.0])), float(rng.choice([6.78e12, 1e9, 14.0]))
        owner, load = plan.partition(world, T, fr, br)
        o_owner, o_load = _oracle_partition(plan, world, T, fr, br)
        assert owner == o_owner
        assert [struct.pack("<d", x) for x in load] == [struct.pack("<d", x) for x in o_load]


@pytest.mark.parametrize("name", ["skinny_74x24x10240", "stacks_experts", "dense_24L", "moe_24L"])
@pytest.mark.parametrize("world", [2, 8])
def test_partition_matches_oracle_on_workloads(muon, name, world):
    import synth
    w = synth.workload(name)
    plan = muon.Plan([(s, w.dtype) for s in w.shapes])
    owner, load = plan.partition(world, w.ns_steps)
    o_owner, o_load = _oracle_partition(plan, world, w.ns_steps, muon.GB300_FLOPS,
                                        muon.GB300_HBM_BYTES)
    assert owner == o_owner and load == o_load
    assert sorted(set(owner)) == list(range(world))


def test_partition_rejects_bad_arguments(muon):
    import torch
    plan = muon.Plan([((24, 64), torch.bfloat16)])
    L = muon.load()
    own = (ctypes.c_int * 1)()
    assert L.muon_plan_partition(plan.handle, 0, 5, 1e15, 1e12, own, None) == -1
    assert L.muon_plan_partition(plan.handle, 2, -1, 1e15, 1e12, own, None) == -1
    assert L.muon_plan_partition(plan.handle, 2, 5, 0.0, 1e12, own, None) == -1
    assert L.muon_plan_partition(plan.handle, 2, 5, 1e15, float("inf"), own, None) == -1
    assert L.muon_plan_partition(plan.handle, 2, 5, 1e15, 1e12, None, None) == -1
    assert L.muon_plan_partition(None, 2, 5, 1e15, 1e12, own, None) == -1
    assert L.muon_plan_partition(plan.handle, 3, 5, 1e15, 1e12, own, None) == 0 and own[0] == 0


def test_partition_with_more_replicas_than_slices(muon):
    import torch
    plan = muon.Plan([((24, 64), torch.bfloat16), ((2, 100, 80), torch.float32)])
    owner, load = plan.partition(8)
    assert len(owner) == 3 and sorted(owner) == [0, 1, 2]
    assert load[3:] == [0.0] * 5 and all(x > 0 for x in load[:3])
    o_owner, o_load = _oracle_partition(plan, 8, 5, muon.GB300_FLOPS, muon.GB300_HBM_BYTES)
    assert owner == o_owner and load == o_load
    part = muon.Partition(plan, 8)
    assert part.owned(7) == [] and part.owned(0) != []


def test_c_program_uses_the_abi(muon, tmp_path):
    # plain C, linked against libmuon.so, host-only calls
    import subprocess
    src = os.path.join(ROOT, "tests", "c_abi_check.c")
    exe = str(tmp_path / "c_abi_check")
    libdir = os.path.dirname(muon.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           src, "-o", exe, "-L", libdir, "-lmuon", "-Wl,-rpath," + libdir])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_muon_with_adamw_routes_parameters(muon):
    # matrices and stacks to Muon, the rest to AdamW grouped by dtype
    import torch
    params = [torch.zeros(24, 64, dtype=torch.bfloat16), torch.zeros(64, dtype=torch.bfloat16),
              torch.zeros(2, 24, 64, dtype=torch.bfloat16), torch.zeros(10),
              torch.zeros(3, dtype=torch.bfloat16)]
    matrix, other, groups = muon.MuonWithAdamW.route(params)
    assert matrix == [0, 2] and other == [1, 3, 4]
    assert groups == {torch.bfloat16: [1, 4], torch.float32: [3]}
    plan = muon.Plan([params[i] for i in matrix])
    assert plan.num_slices == 3


def test_skinny_plans_fit_the_cluster_tensor_memory(muon):
    # V is held in bf16 in tensor memory between the passes: the slice (rows
    # padded to a block of 8, columns to 32) must fit the cluster's CTAs,
    # each with 128 lanes x 512 columns x 4 bytes; clusters are portable (<= 8)
    import torch
    tmem_cta = 128 * 512 * 4
    for m_ in list(range(1, 65, 3)) + [64]:
        for n_ in (m_, 77, 1000, 10240, 40000, 65536, 100000, 200000):
            if n_ < m_:
                continue
            plan = muon.Plan([((m_, n_), torch.bfloat16)])
            (g,) = plan.groups()
            if g["kernel"] != muon.KERNEL_SKINNY:
                continue
            mp8 = (m_ + 7) // 8 * 8
            n32 = (n_ + 31) // 32 * 32
            assert 1 <= g["cluster"] <= 8, (m_, n_)
            assert mp8 * n32 * 2 <= g["cluster"] * tmem_cta, (m_, n_, g["cluster"])
    # a slice too long for 8 CTAs goes to the dense path
    (g,) = muon.Plan([((64, 1 << 20), torch.bfloat16)]).groups()
    assert g["kernel"] == muon.KERNEL_DENSE


def test_alloc_host_errors_on_the_host(muon):
    # no element, or (on a machine without a device) a registration the
    # driver refuses: an error, and nothing is held
    import torch
    with pytest.raises(ValueError):
        muon.alloc_host(0, torch.float32)
    if not torch.cuda.is_available():
        with pytest.raises(muon.MuonError) as e:
            muon.alloc_host(1024, torch.float32)
        assert e.value.status == -5
    L = muon.load()
    assert L.muon_host_free(None) == 0
    assert L.muon_host_free(ctypes.c_void_p(0x123000)) == -1
