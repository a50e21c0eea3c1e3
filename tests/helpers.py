"""Shared helpers of the GPU parity tests: run libmuon on seeded inputs and
compare with the fp64 oracle on the same host bytes.

Tolerances (fixed for the Muon step):
  * O, per slice: relative Frobenius error <= 2e-2 in the fp16 tensor-core
    mode and <= 1e-4 in the fp32 mode;
  * momentum: |M'_gpu - M'_oracle| <= 1e-6 * (beta |M| + |G|) elementwise
    (one fp32 multiply-add of fp64-exact inputs);
  * bf16 parameters: (1) within one bf16 ulp of the round-to-nearest-even
    value of W*(1 - lr*wd) - lr*s*O_gpu (the update applied to the GPU's own
    O), and (2) within one ulp of the oracle's W' plus lr*s*|O_gpu - O_oracle|
    (a parameter near zero carries the O error at more than one ulp of its
    own size); fp32 parameters: relative Frobenius error of W' - W within
    the O tolerance.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import synth

TOL = {"tc16": 2e-2, "fp32": 1e-4}
HOST_THREADS = max(1, min(32, os.cpu_count() or 1))


def muon():
    from newton_schulz_05_gb300 import build
    build.build()
    import newton_schulz_05_gb300 as m
    m.load()
    return m


def slices(t):
    return [t] if t.dim() == 2 else [t[e] for e in range(t.shape[0])]


def make_inputs(shapes, dtype, grad_std=1e-2, seed=0, steps=1, device="cpu", param_std=0.02):
    W = [synth.draw(s, param_std, synth.param_seed(1, i), dtype, device) for i, s in enumerate(shapes)]
    Gs = [[synth.draw(s, grad_std, synth.param_seed(seed + t, i), dtype, device)
           for i, s in enumerate(shapes)] for t in range(steps)]
    M = [torch.zeros(s, dtype=torch.float32, device=device) for s in shapes]
    return W, Gs, M


def gpu_step(plan, W, G, M, hp, ortho=True, ws=None):
    """One step on the GPU.  W, G, M: lists of CUDA tensors (updated in place
    for W and M).  Returns the list of O tensors (or None)."""
    m = muon()
    if ws is None:
        ws = m.alloc_workspace(plan)
    O = [torch.empty(w.shape, dtype=torch.float32, device=w.device) for w in W] if ortho else None
    m.step(plan, W, G, M, lr=hp["lr"], beta=hp["beta"], wd=hp["wd"], nesterov=hp["nesterov"],
           ns_steps=hp["ns_steps"], coeffs=hp.get("coeffs", synth.Workload("", (), torch.float32, 1).coeffs),
           workspace=ws, ortho=O)
    torch.cuda.synchronize()
    assert m.workspace_error(ws) == 0
    return O


def update_scale(M, N, hp):
    """Update scale s of a [M, N] slice (float32 value), by hp's scale_mode."""
    if hp.get("scale_mode", "sqrt_ratio") == "rms_match":
        return float(np.float32(0.2 * np.sqrt(max(M, N))))
    return float(np.float32(np.sqrt(max(1.0, M / N))))


def oracle_step(W, G, M, hp, which=None):
    """fp64 oracle over the slices of W/G/M (CPU tensors).  `which` selects
    (param, slice) pairs; default all.  Returns {(p, e): (W', M', O)}."""
    keys, ws, gs, ms = [], [], [], []
    for p in range(len(W)):
        sw, sg, sm = slices(W[p]), slices(G[p]), slices(M[p])
        for e in range(len(sw)):
            if which is not None and (p, e) not in which:
                continue
            keys.append((p, e)); ws.append(sw[e]); gs.append(sg[e]); ms.append(sm[e])
    threads = HOST_THREADS
    if len(keys) < threads or max(w.numel() for w in ws) > (1 << 20):
        # few or big slices: one at a time, each spread over the host threads
        out = {}
        for k, w, g, mm in zip(keys, ws, gs, ms):
            out[k] = oracle.muon_slice(w, g, mm, hp["lr"], hp["beta"], hp["wd"], hp["nesterov"],
                                       T=hp["ns_steps"],
                                       coeffs=hp.get("coeffs", oracle.DEFAULT_COEFFS),
                                       scale=update_scale(*w.shape, hp), threads=threads)
        return out
    wo, mo, oo, _ = oracle.muon_slices(ws, gs, ms, hp["lr"], hp["beta"], hp["wd"], hp["nesterov"],
                                       T=hp["ns_steps"], coeffs=hp.get("coeffs", oracle.DEFAULT_COEFFS),
                                       scales=[update_scale(*w.shape, hp) for w in ws],
                                       threads=threads)
    return {k: (wo[i], mo[i], oo[i]) for i, k in enumerate(keys)}


def rel_fro(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    nb = np.sqrt((b * b).sum())
    d = np.sqrt(((a - b) ** 2).sum())
    if nb == 0:
        return 0.0 if d == 0 else float("inf")
    return d / nb


def bf16_ulp(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    return np.where(x > 0, 2.0 ** (e - 7), 2.0 ** -133)


def compare(key, gpu, ref, W0, G, M0, hp, mode, dtype, report=None):
    """Assert one slice's GPU results against the oracle's."""
    Wg, Mg, Og = [np.asarray(x.double().cpu().numpy(), np.float64) for x in gpu]
    Wr, Mr, Or = ref
    W0 = np.asarray(W0.double().cpu().numpy()); G = np.asarray(G.double().cpu().numpy())
    M0 = np.asarray(M0.double().cpu().numpy())
    tol = TOL[mode]
    if Og is not None:
        e = rel_fro(Og, Or)
        if report is not None:
            report.append((key, e))
        assert e <= tol, "slice %s: O relative error %.3g > %.1g" % (key, e, tol)
    bound = 1e-6 * (hp["beta"] * np.abs(M0) + np.abs(G)) + 1e-30
    assert np.all(np.abs(Mg - Mr) <= bound), "slice %s: momentum mismatch" % (key,)
    if dtype == torch.bfloat16:
        # (1) the update arithmetic on the GPU's own O: W' is the RNE rounding
        #     of W*(1 - lr*wd) - lr*s*O within one bf16 ulp (fp32 intermediates)
        M_, N_ = W0.shape
        s = update_scale(M_, N_, hp)
        own = W0 * (1 - hp["lr"] * hp["wd"]) - hp["lr"] * s * Og
        own_b = torch.from_numpy(own).to(torch.bfloat16).double().numpy()
        # fp32 intermediates (decay, lr*s, the product) round at 2^-24 of
        # the terms; this matters where the two terms cancel
        terms = np.abs(W0 * (1 - hp["lr"] * hp["wd"])) + hp["lr"] * s * np.abs(Og)
        ulp = np.maximum(bf16_ulp(own_b), bf16_ulp(Wg)) + 4 * 2.0 ** -24 * terms
        bad = np.abs(Wg - own_b) > ulp
        assert not bad.any(), "slice %s: %d params off the update of the GPU's O" % (key, int(bad.sum()))
        # (2) against the oracle: one ulp of its W' plus the O difference
        #     carried through the update, lr*s*|O_gpu - O_oracle|
        Wr_b = torch.from_numpy(Wr).to(torch.bfloat16).double().numpy()
        ulp = np.maximum(bf16_ulp(Wr_b), bf16_ulp(Wg))
        bound = ulp + hp["lr"] * s * np.abs(Og - Or) * 1.001 + 4 * 2.0 ** -24 * terms
        bad = np.abs(Wg - Wr_b) > bound
        assert not bad.any(), "slice %s: %d params beyond the bf16 bound" % (key, int(bad.sum()))
    else:
        e = rel_fro(Wg - W0, Wr - W0)
        assert e <= tol, "slice %s: W'-W relative error %.3g" % (key, e)


def run_and_check(shapes, dtype, hp, mode="tc16", grad_std=1e-2, seed=0, which=None,
                  skinny_max_m=64, report=None):
    """Seeded inputs -> GPU step (with O) and oracle -> compare every (or the
    selected) slice.  Returns the plan."""
    m = muon()
    W, Gs, M = make_inputs(shapes, dtype, grad_std=grad_std, seed=seed)
    G = Gs[0]
    plan = m.Plan([(tuple(s), dtype) for s in shapes], mode=mode, skinny_max_m=skinny_max_m,
                  scale_mode=hp.get("scale_mode", "sqrt_ratio"))
    Wd = [w.cuda() for w in W]; Gd = [g.cuda() for g in G]; Md = [x.cuda() for x in M]
    O = gpu_step(plan, Wd, Gd, Md, hp)
    ref = oracle_step(W, G, M, hp, which)
    for (p, e), r in ref.items():
        gp = (slices(Wd[p])[e], slices(Md[p])[e], slices(O[p])[e])
        compare((p, e), gp, r, slices(W[p])[e], slices(G[p])[e], slices(M[p])[e], hp, mode, dtype,
                report)
    return plan


def compare_folded(key, Wf, W0, G, M0, Og, ref, hp, dtype):
    """Assert one slice's parameters from the step WITHOUT an O output
    against the oracle, element by element.

    On the fused skinny kernel that step folds the update factor -lr*s into
    the 16-bit left operand of its last product: it computes
    sum_k RNE16(-lr*s*Q~_ik) V_kj instead of -lr*s * sum_k RNE16(Q~_ik) V_kj,
    with Q~ = Q/(||V|| + eps) and O = Q X0.  bf16 keeps 8 significant bits,
    so one round-to-nearest moves a value by at most 2^-8 of itself; the two
    left operands are rounded separately, so they differ by at most 2^-7
    relative per entry, and the update term differs from the one of the step
    that writes O (Og, same kernel, same V and fp32 Q bits) by at most
    lr*s*2^-7*(|Q| |X0|)_ij.  Q is recovered from the oracle in fp64 as
    the m x m matrix with O = Q X0 (X0 has full row rank).  The bound per
    parameter, against the round-to-nearest value of the oracle's W':
      ulp + lr*s*|Og - O_oracle| + 1.05 * lr*s*2^-7*(|Q| |X0|) + 4*2^-24*terms
    (the 5% covers the fp32 Q of the kernel against the fp64 one).  On the
    dense path the step without O is the same arithmetic as the one with O,
    so there the last two terms of the bound are not needed (the tests check
    those parameters bit for bit against the O-writing step as well)."""
    Wf = np.asarray(Wf.double().cpu().numpy(), np.float64)
    W0 = np.asarray(W0.double().cpu().numpy(), np.float64)
    G = np.asarray(G.double().cpu().numpy(), np.float64)
    M0 = np.asarray(M0.double().cpu().numpy(), np.float64)
    Og = np.asarray(Og.double().cpu().numpy(), np.float64)
    Wr, _, Or = ref
    M_, N_ = W0.shape
    s = update_scale(M_, N_, hp)
    lrs = hp["lr"] * s
    Mp = hp["beta"] * M0 + G
    V = G + hp["beta"] * Mp if hp["nesterov"] else Mp
    X0 = V / (np.linalg.norm(V) + 1e-7)
    Xw, Ow = (X0.T, Or.T) if M_ > N_ else (X0, Or)
    # O = Q X0  ->  Q = O X0^T (X0 X0^T)^-1   (working orientation, m x m)
    Q = np.linalg.solve(Xw @ Xw.T, Xw @ Ow.T).T
    qx = np.abs(Q) @ np.abs(Xw)
    if M_ > N_:
        qx = qx.T
    terms = np.abs(W0 * (1 - hp["lr"] * hp["wd"])) + lrs * np.abs(Og)
    if dtype == torch.bfloat16:
        Wr_r = torch.from_numpy(Wr).to(torch.bfloat16).double().numpy()
        ulp = np.maximum(bf16_ulp(Wr_r), bf16_ulp(Wf))
    else:
        Wr_r = Wr.astype(np.float32).astype(np.float64)
        ulp = np.maximum(np.spacing(np.abs(Wr_r).astype(np.float32)),
                         np.spacing(np.abs(Wf).astype(np.float32))).astype(np.float64)
    fold = 1.05 * lrs * 2.0 ** -7 * qx
    bound = ulp + lrs * np.abs(Og - Or) * 1.001 + fold + 4 * 2.0 ** -24 * terms
    diff = np.abs(Wf - Wr_r)
    bad = diff > bound
    if bad.any():
        i = np.unravel_index(np.argmax(diff - bound), diff.shape)
        raise AssertionError(
            "slice %s: %d params of the step without O beyond the bound; worst at %s: "
            "|W' - W'_oracle| %.3g, bound %.3g (ulp %.3g, O term %.3g, fold term %.3g)" % (
                key, int(bad.sum()), i, diff[i], bound[i], ulp[i],
                lrs * abs(Og[i] - Or[i]), fold[i]))
