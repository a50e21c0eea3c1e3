"""muon_adamw_step: AdamW for the parameters Muon does not orthogonalise
(1-D biases and norm scales, and any other tensor kept off the Muon path),
one launch for many tensors, against the fp64 oracle element by element.

Tolerances: moments within 1e-6 of the magnitudes of their two terms (fp32
storage of fp64 math; the terms of m' can cancel);
parameters within one ulp of the oracle's W' (bf16 round-to-nearest-even)
plus 4 * 2^-24 of |W (1 - lr wd)| + lr |m-terms| / (sqrt(v_hat) + eps) (fp32
intermediates: where the two terms of m' cancel, its fp32 error is relative
to the terms, and it reaches W' through the update), for fp32 parameters the
same bound in fp32 ulps.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_ulp, muon

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1)
# the hyper-parameters as the library receives them (fp32 through the C ABI):
# 1 - beta2 of the float 0.999 is 1.3e-5 away from 1e-3
HP32 = {k: float(np.float32(v)) for k, v in HP.items()}
SIZES = [1, 3, 24, 1000, 4096, 4097, 10240, 70001, 2 * 4096 * 3 + 5]


def _run(dtype, steps=3, sizes=SIZES):
    m = muon()
    W = [synth.draw((n,), 0.02, synth.param_seed(1, i), dtype) for i, n in enumerate(sizes)]
    Gs = [[synth.draw((n,), 1e-2, synth.param_seed(10 + t, i), dtype) for i, n in enumerate(sizes)]
          for t in range(steps)]
    Wd = [w.cuda() for w in W]
    Md = [torch.zeros(n, device="cuda") for n in sizes]
    Vd = [torch.zeros(n, device="cuda") for n in sizes]
    Wr = [w.double().numpy() for w in W]
    Mr = [np.zeros(n) for n in sizes]
    Vr = [np.zeros(n) for n in sizes]
    for t in range(1, steps + 1):
        G = Gs[t - 1]
        W0 = [w.cpu() for w in Wd]
        m.adamw_step(Wd, [g.cuda() for g in G], Md, Vd, step=t, **HP)
        torch.cuda.synchronize()
        for i in range(len(sizes)):
            # teacher-forced: the oracle starts from the GPU's state of step t-1
            wo, mo, vo = oracle.adamw(W0[i], G[i], Mr[i], Vr[i], HP32["lr"], HP32["beta1"],
                                      HP32["beta2"], HP32["eps"], HP32["wd"], t)
            mg = Md[i].double().cpu().numpy(); vg = Vd[i].double().cpu().numpy()
            # the two terms of m' can cancel: bound by their magnitudes
            gd = G[i].double().numpy()
            mbound = 1e-6 * (HP32["beta1"] * np.abs(Mr[i]) + (1 - HP32["beta1"]) * np.abs(gd)) + 1e-30
            assert np.all(np.abs(mg - mo) <= mbound), (t, i)
            assert np.all(np.abs(vg - vo) <= 1e-6 * np.abs(vo) + 1e-38), (t, i)
            wg = Wd[i].double().cpu().numpy()
            w0 = W0[i].double().numpy()
            upd = np.abs(wo - w0 * (1 - HP["lr"] * HP["wd"]))
            inv_c1 = 1.0 / (1.0 - HP32["beta1"] ** t)
            inv_c2 = 1.0 / (1.0 - HP32["beta2"] ** t)
            uterm = HP32["lr"] * inv_c1 * (mbound * 1e6) / (np.sqrt(vo * inv_c2) + HP32["eps"])
            slack = 4 * 2.0 ** -24 * (np.abs(w0) + upd + uterm)
            if dtype == torch.bfloat16:
                wr = torch.from_numpy(wo).to(torch.bfloat16).double().numpy()
                ulp = np.maximum(bf16_ulp(wr), bf16_ulp(wg))
            else:
                wr = wo
                ulp = np.spacing(np.abs(wo).astype(np.float32)).astype(np.float64)
            assert np.all(np.abs(wg - wr) <= ulp + slack), (t, i)
            Mr[i], Vr[i] = mg, vg


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_adamw_matches_oracle(dtype):
    _run(dtype)


def test_adamw_many_tensors_in_several_launches():
    # more than 256 tensors: the launch is split, results are unchanged
    _run(torch.bfloat16, steps=1, sizes=[(i % 7) * 97 + 1 for i in range(300)])


def test_adamw_zero_lr_keeps_params():
    m = muon()
    W = [torch.randn(n, device="cuda").bfloat16() for n in (5, 1000)]
    W0 = [w.clone() for w in W]
    m.adamw_step(W, [torch.randn_like(w) for w in W], [torch.zeros(w.numel(), device="cuda") for w in W],
                 [torch.zeros(w.numel(), device="cuda") for w in W], lr=0.0, wd=0.1, step=1)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(W, W0))


def test_muon_with_adamw_equals_the_separate_steps():
    # one MuonWithAdamW step == Muon on the matrices + AdamW on the rest, bit for bit
    m = muon()
    shapes = [(24, 1000), (300,), (2, 200, 150), (77,), (5,)]
    dts = [torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.float32, torch.bfloat16]
    P = [synth.draw(s, 0.02, synth.param_seed(1, i), d, "cuda") for i, (s, d) in enumerate(zip(shapes, dts))]
    G = [synth.draw(s, 1e-2, synth.param_seed(2, i), d, "cuda") for i, (s, d) in enumerate(zip(shapes, dts))]
    P2 = [p.clone() for p in P]
    opt = m.MuonWithAdamW(P, adamw_lr=1e-3, adamw_wd=0.01)
    for _ in range(2):
        opt.step(G)
    ref_muon = m.Muon([P2[0], P2[2]])
    mom = {i: (torch.zeros(P2[i].numel(), device="cuda"), torch.zeros(P2[i].numel(), device="cuda"))
           for i in (1, 3, 4)}
    for t in (1, 2):
        ref_muon.step([G[0], G[2]])
        for idx in ([1, 4], [3]):
            m.adamw_step([P2[i].view(-1) for i in idx], [G[i].reshape(-1) for i in idx],
                         [mom[i][0] for i in idx], [mom[i][1] for i in idx], lr=1e-3, wd=0.01, step=t)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(P, P2))
