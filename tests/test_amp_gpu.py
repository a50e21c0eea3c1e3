"""muon_step_amp: the step on loss-scaled gradients (mixed-precision training
behind a loss scaler, as in the Paddle Muon sharding PR's AMP GradScaler
path).  Against the oracle's loss-scaled step and against muon_step:
  * a power-of-two inv_scale is exact in both dtypes, so the step on S*G with
    inv_scale 1/S equals muon_step on G bit for bit;
  * one inf or NaN anywhere skips the whole step: found_inf = 1 and every
    parameter and momentum buffer keeps its bits;
  * any other inv_scale matches the oracle within the usual tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import compare, gpu_step, make_inputs, muon, slices

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5, coeffs=oracle.DEFAULT_COEFFS)
SHAPES = [(24, 700), (2, 24, 1024), (200, 300), (300, 200)]


def _amp(plan, W, G, M, inv_scale, ws=None):
    m = muon()
    ws = m.alloc_workspace(plan) if ws is None else ws
    found = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    m.step_amp(plan, W, G, M, lr=HP["lr"], beta=HP["beta"], wd=HP["wd"], inv_scale=inv_scale,
               found_inf=found, nesterov=HP["nesterov"], ns_steps=HP["ns_steps"],
               coeffs=HP["coeffs"], workspace=ws)
    torch.cuda.synchronize()
    assert m.workspace_error(ws) == 0
    return int(found.item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_power_of_two_scale_equals_plain_step(dtype):
    m = muon()
    W, Gs, M = make_inputs(SHAPES, dtype)
    plan = m.Plan([(s, dtype) for s in SHAPES])
    Wa = [w.cuda() for w in W]; Ma = [x.cuda() for x in M]
    gpu_step(plan, Wa, [g.cuda() for g in Gs[0]], Ma, HP, ortho=False)
    S = 2.0 ** 10
    Wb = [w.cuda() for w in W]; Mb = [x.cuda() for x in M]
    Gs_scaled = [(g.float() * S).to(dtype).cuda() for g in Gs[0]]
    assert all(torch.equal(a.cpu().float() / S, b.float()) for a, b in zip(Gs_scaled, Gs[0]))
    assert _amp(plan, Wb, Gs_scaled, Mb, 1.0 / S) == 0
    assert all(torch.equal(a, b) for a, b in zip(Wa, Wb))
    assert all(torch.equal(a, b) for a, b in zip(Ma, Mb))


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")], ids=["inf", "-inf", "nan"])
@pytest.mark.parametrize("where", [0, 1, 2, 3])
def test_non_finite_gradient_skips_the_whole_step(bad, where):
    m = muon()
    W, Gs, M = make_inputs(SHAPES, torch.bfloat16)
    M = [torch.randn(x.shape, generator=torch.Generator().manual_seed(5)) for x in M]
    plan = m.Plan([(s, torch.bfloat16) for s in SHAPES])
    G = [g.clone() for g in Gs[0]]
    flat = G[where].view(-1)
    flat[flat.numel() // 3] = bad
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    assert _amp(plan, Wd, [g.cuda() for g in G], Md, 0.25) == 1
    assert all(torch.equal(a.cpu(), b) for a, b in zip(Wd, W))
    assert all(torch.equal(a.cpu(), b) for a, b in zip(Md, M))
    # the next clean step runs and clears the flag
    assert _amp(plan, Wd, [g.cuda() for g in Gs[0]], Md, 0.25) == 0
    assert not torch.equal(Wd[0].cpu(), W[0])


def test_general_scale_matches_oracle():
    m = muon()
    W, Gs, M = make_inputs(SHAPES, torch.bfloat16, grad_std=30.0)
    plan = m.Plan([(s, torch.bfloat16) for s in SHAPES])
    inv = 1.0 / 3000.7
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    assert _amp(plan, Wd, [g.cuda() for g in Gs[0]], Md, inv) == 0
    ws_, gs_, ms_, keys = [], [], [], []
    for p in range(len(W)):
        for e, (w, g, mo) in enumerate(zip(slices(W[p]), slices(Gs[0][p]), slices(M[p]))):
            ws_.append(w); gs_.append(g); ms_.append(mo); keys.append((p, e))
    wo, mo_, oo, found = oracle.muon_slices_amp(ws_, gs_, ms_, HP["lr"], HP["beta"], HP["wd"],
                                                HP["nesterov"], inv, threads=8)
    assert not found
    for i, (p, e) in enumerate(keys):
        wg = slices(Wd[p])[e].cpu(); mg = slices(Md[p])[e].cpu()
        # no O from this entry point: check W through the bf16 bound with the
        # oracle's own O, and the momentum tightly
        Mr = mo_[i]
        gu = np.abs(gs_[i].double().numpy()) * inv
        assert np.all(np.abs(mg.double().numpy() - Mr) <=
                      1e-6 * (0.95 * np.abs(slices(M[p])[e].double().numpy()) + gu) + 1e-30)
        d = np.abs(wg.double().numpy() - torch.from_numpy(wo[i]).to(torch.bfloat16).double().numpy())
        # one bf16 ulp plus lr*s*2e-2 of |O| (the O tolerance carried through the update)
        s = float(np.float32(np.sqrt(max(1.0, wg.shape[0] / wg.shape[1]))))
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(wo[i]), 1e-30))) - 7)
        assert np.all(d <= ulp + HP["lr"] * s * 2e-2 * np.abs(oo[i]).max() + 1e-12)
