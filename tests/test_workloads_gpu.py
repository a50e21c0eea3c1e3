"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times: one muon_step over every parameter,
without O outputs (the benchmark's own call, PreparedStep), and beside it
muon_step_ortho on identical inputs so that O itself meets the oracle.

  * fp32 [24, 1024]: every slice against the oracle;
  * 74 x [24, 10240], 10 steps, teacher-forced (the oracle's step t+1
    starts from the GPU's state after step t, so errors do not compound):
    every slice of both calls, every step, element by element;
  * stacks + experts, MoE model, dense layers: both calls over the whole
    workload; momentum of the two calls bit for bit, dense-group parameters
    bit for bit; every slice of the skinny groups and the first and last
    slice of every other group against the oracle, element by element
    (the dense layers' [11008, 4096] group is worked on transposed);
  * every dense group at full size against the closed form of Newton-Schulz
    on a Householder-structured input (a property that holds at any size).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, compare, compare_folded, gpu_step, muon, oracle_step, slices

pytestmark = pytest.mark.gpu


def hp_of(w):
    return dict(lr=w.lr, beta=w.beta, wd=w.wd, nesterov=w.nesterov, ns_steps=w.ns_steps,
                coeffs=w.coeffs)


def test_fp32_24x1024_full():
    w = synth.workload("fp32_24x1024")
    m = muon()
    W = synth.make_params(w); G = synth.make_grads(w, 0); M = synth.make_momentum(w)
    plan = m.Plan(list(zip(w.shapes, [w.dtype] * len(w.shapes))))
    Wd = [x.cuda() for x in W]; Md = [x.cuda() for x in M]
    O = gpu_step(plan, Wd, [g.cuda() for g in G], Md, hp_of(w))
    ref = oracle_step(W, G, M, hp_of(w))
    for (p, e), r in ref.items():
        compare((p, e), (Wd[p].cpu(), Md[p].cpu(), O[p].cpu()), r, W[p], G[p], M[p], hp_of(w),
                "tc16", w.dtype)


def _both_paths(plan, W, G, M, hp):
    """The benchmark's call (PreparedStep, no O) on (W, G, M) in place, and
    muon_step_ortho on copies of W and M.  Returns (W copy, M copy, O)."""
    m = muon()
    Wb = [x.clone() for x in W]; Mb = [x.clone() for x in M]
    O = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in W]
    ws = m.alloc_workspace(plan, W[0].device)
    m.PreparedStep(plan, W, G, M, workspace=ws, **hp)()
    torch.cuda.synchronize()
    assert m.workspace_error(ws) == 0
    m.step(plan, Wb, G, Mb, workspace=ws, ortho=O, **hp)
    torch.cuda.synchronize()
    assert m.workspace_error(ws) == 0
    del ws
    return Wb, Mb, O


def test_skinny_74x24x10240_ten_steps_bench_call_teacher_forced():
    w = synth.workload("skinny_74x24x10240")
    m = muon()
    hp = hp_of(w)
    plan = m.Plan(list(zip(w.shapes, [w.dtype] * len(w.shapes))))
    Wd = [x.cuda() for x in synth.make_params(w)]
    Md = [x.cuda() for x in synth.make_momentum(w)]
    for t in range(w.steps):
        G = synth.make_grads(w, t)
        W0 = [x.cpu() for x in Wd]; M0 = [x.cpu() for x in Md]
        Wb, Mb, O = _both_paths(plan, Wd, [g.cuda() for g in G], Md, hp)
        ref = oracle_step(W0, G, M0, hp)
        for p in range(len(Wd)):
            assert torch.equal(Md[p], Mb[p]), (t, p)
            r = ref[(p, 0)]
            og = O[p].cpu()
            compare((t, p), (Wb[p].cpu(), Mb[p].cpu(), og), r, W0[p], G[p], M0[p], hp, "tc16",
                    w.dtype)
            compare_folded((t, p), Wd[p].cpu(), W0[p], G[p], M0[p], og, r, hp, w.dtype)


def _sampled_keys(plan, shapes):
    """(param, slice) pairs: all slices of skinny groups, first and last of
    the others."""
    mm = muon()
    groups = plan.groups()
    members = {g: [] for g in range(len(groups))}
    for p, s in enumerate(shapes):
        for e in range(s[0] if len(s) == 3 else 1):
            g, i = plan.slice(p, e)
            members[g].append((p, e))
    keys = set()
    for g, lst in members.items():
        if groups[g]["kernel"] == mm.KERNEL_SKINNY:
            keys.update(lst)
        else:
            keys.update([lst[0], lst[-1]])
    return keys, groups


def _run_workload(name, keep=lambda key, group: True):
    w = synth.workload(name)
    m = muon()
    hp = hp_of(w)
    shapes = list(w.shapes)
    plan = m.Plan(list(zip(shapes, [w.dtype] * len(shapes))))
    W = synth.make_params(w, device="cuda")
    G = synth.make_grads(w, 0, device="cuda")
    M = synth.make_momentum(w, device="cuda")
    keys, groups = _sampled_keys(plan, shapes)
    keys = sorted(k for k in keys if keep(k, groups[plan.slice(*k)[0]]))
    W0 = {k: slices(W[k[0]])[k[1]].cpu() for k in keys}
    G0 = {k: slices(G[k[0]])[k[1]].cpu() for k in keys}
    M0 = {k: slices(M[k[0]])[k[1]].cpu() for k in keys}
    Wb, Mb, O = _both_paths(plan, W, G, M, hp)
    # the two calls: momentum bit for bit; dense-group parameters bit for bit
    for p in range(len(shapes)):
        assert torch.equal(M[p], Mb[p]), p
        if groups[plan.slice(p, 0)[0]]["kernel"] == m.KERNEL_DENSE:
            assert torch.equal(W[p], Wb[p]), p
    errs = []
    # oracle per group, so one big slice spreads over all host threads
    for g in range(len(groups)):
        ks = [k for k in keys if plan.slice(*k)[0] == g]
        if not ks:
            continue
        ref = oracle_step([W0[k] for k in ks], [G0[k] for k in ks], [M0[k] for k in ks], hp)
        for j, k in enumerate(ks):
            og = slices(O[k[0]])[k[1]].cpu()
            compare(k, (slices(Wb[k[0]])[k[1]].cpu(), slices(Mb[k[0]])[k[1]].cpu(), og),
                    ref[(j, 0)], W0[k], G0[k], M0[k], hp, "tc16", w.dtype, errs)
            if groups[g]["kernel"] == m.KERNEL_SKINNY:
                compare_folded(k, slices(W[k[0]])[k[1]].cpu(), W0[k], G0[k], M0[k], og,
                               ref[(j, 0)], hp, w.dtype)
    return errs


def test_stacks_and_experts():
    errs = _run_workload("stacks_experts")
    assert len(errs) == 256 + 4


def test_moe_model_sampled_slices():
    errs = _run_workload("moe_24L")
    assert len(errs) == 74 + 2 * 3


def test_dense_layers_bench_call():
    # the benchmark's default workload: 24 x {4 x [4096, 4096], [11008, 4096],
    # 2 x [4096, 11008]}; the oracle takes the first and last slice of the two
    # [*, 11008] groups (one worked on transposed) and the first [4096, 4096]
    def keep(key, group):
        return not (group["M"] == 4096 and group["N"] == 4096 and key[0] != 0)
    errs = _run_workload("dense_24L", keep)
    assert len(errs) == 5


def _p_scalar(x, T, coeffs):
    a, b, c = coeffs
    for _ in range(T):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def _householder_case(M, N, seed):
    """V = (I - 2uu^T) D (I - 2ww^T) with D rectangular diagonal, and the
    exact Newton-Schulz result O = (I - 2uu^T) p^T(D / (||d|| + eps)) (I - 2ww^T)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    k = min(M, N)
    u = torch.randn(M, generator=gen, dtype=torch.float64); u /= u.norm()
    v = torch.randn(N, generator=gen, dtype=torch.float64); v /= v.norm()
    d = 0.2 + 0.8 * torch.rand(k, generator=gen, dtype=torch.float64)
    return u, v, d


def _rect_from_diag(u, v, diag, M, N, dev):
    """(I - 2uu^T) R (I - 2vv^T) for R = rectangular diag(diag), on `dev`."""
    u = u.to(dev); v = v.to(dev); diag = diag.to(dev)
    k = diag.numel()
    R = torch.zeros(M, N, dtype=torch.float64, device=dev)
    R[torch.arange(k), torch.arange(k)] = diag
    a = torch.zeros(N, dtype=torch.float64, device=dev); a[:k] = diag * u[:k]   # R^T u
    b = torch.zeros(M, dtype=torch.float64, device=dev); b[:k] = diag * v[:k]   # R v
    gamma = (u[:k] * diag * v[:k]).sum()
    return R - 2 * torch.outer(u, a) - 2 * torch.outer(b, v) + 4 * gamma * torch.outer(u, v)


@pytest.mark.parametrize("shape", [(4096, 4096), (11008, 4096), (4096, 11008), (2048, 2048),
                                   (1408, 2048), (2048, 1408)], ids=str)
def test_dense_groups_householder_closed_form(shape):
    m = muon()
    M_, N_ = shape
    u, v, d = _householder_case(M_, N_, seed=M_ * 7 + N_)
    V = _rect_from_diag(u, v, d, M_, N_, "cuda")
    G = V.float().contiguous()
    W = torch.zeros(shape, dtype=torch.float32, device="cuda")
    Mom = torch.zeros(shape, dtype=torch.float32, device="cuda")
    plan = m.Plan([(shape, torch.float32)])
    hp = dict(lr=0.02, beta=0.0, wd=0.0, nesterov=False, ns_steps=5, coeffs=oracle.DEFAULT_COEFFS)
    O = gpu_step(plan, [W], [G], [Mom], hp)[0]
    nd = float(d.norm())
    p = _p_scalar(d / (nd + 1e-7), 5, oracle.DEFAULT_COEFFS)
    Oe = _rect_from_diag(u, v, p, M_, N_, "cuda")
    err = float((O.double() - Oe).norm() / Oe.norm())
    assert err <= TOL["tc16"], err
    # the update is W' = 0 - lr * s * O exactly as computed from O
    s = float(np.float32(np.sqrt(max(1.0, M_ / N_))))
    assert float((W.double() + 0.02 * s * O.double()).abs().max()) < 1e-6
