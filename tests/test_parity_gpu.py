"""GPU parity: libmuon (through the C ABI) against the fp64 oracle, element
by element on seeded inputs, plus exact properties of the step.

Sizes span several tiles and ragged tails on both kernel families: the fused
on-chip kernel (min(M,N) <= 64) and the dense path; both 2D and 3D stacks,
M < N and M > N (transposed), both parameter dtypes and both arithmetic
modes.  Workload-size cases live in test_workloads_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (TOL, compare, gpu_step, make_inputs, muon, oracle_step, rel_fro,
                     run_and_check, slices)

pytestmark = pytest.mark.gpu

HP = dict(lr=0.02, beta=0.95, wd=0.1, nesterov=True, ns_steps=5, coeffs=oracle.DEFAULT_COEFFS)


def test_fp32_single_matrix_24x1024_both_modes():
    # one fp32 [24, 1024] parameter, grad ~ N(0, 1) seed 0, beta 0.95 Nesterov,
    # 5 steps, lr 0.02, wd 0.1, a single step from zero momentum
    for mode in ("tc16", "fp32"):
        run_and_check([(24, 1024)], torch.float32, HP, mode=mode, grad_std=1.0)


# m covers every row-block count of the fused kernel (1, 2, 3, 4, 6, 8 blocks
# of 8 rows), with n a multiple of 8 (rows streamed through the shared-memory
# ring) and not (direct loads), and both orientations
SKINNY = [(24, 1024), (24, 10240), (5, 77), (64, 300), (20, 33), (1, 1), (1, 500), (500, 1),
          (8, 8), (40, 2000), (56, 130), (1000, 24), (300, 64), (17, 4099), (3, 24, 500),
          (12, 3000), (16, 520), (32, 2048), (30, 1000), (2000, 12)]


@pytest.mark.parametrize("shape", SKINNY, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_skinny_kernel_matches_oracle(shape, dtype):
    plan = run_and_check([shape], dtype, HP)
    assert plan.groups()[0]["kernel"] == muon().KERNEL_SKINNY


DENSE = [(130, 260), (256, 384), (300, 200), (65, 1000), (2, 200, 150), (128, 128), (129, 129),
         (1000, 70)]


@pytest.mark.parametrize("shape", DENSE, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", ["tc16", "fp32"])
def test_dense_path_matches_oracle(shape, mode):
    plan = run_and_check([shape], torch.bfloat16, HP, mode=mode)
    assert plan.groups()[0]["kernel"] == muon().KERNEL_DENSE


@pytest.mark.parametrize("shape", [(24, 1024), (3, 40, 300), (500, 24)], ids=str)
def test_fp32_mode_on_skinny_shapes(shape):
    plan = run_and_check([shape], torch.float32, HP, mode="fp32")
    assert plan.groups()[0]["kernel"] == muon().KERNEL_DENSE


def test_mixed_groups_one_call():
    shapes = [(24, 700), (2, 24, 700), (200, 150), (150, 200), (700, 24), (24, 700)]
    plan = run_and_check(shapes, torch.bfloat16, HP)
    kinds = [g["kernel"] for g in plan.groups()]
    assert len(kinds) == 4 and plan.groups()[0]["count"] == 4


@pytest.mark.parametrize("shape", [(24, 1000), (200, 300)], ids=str)
@pytest.mark.parametrize("T", [0, 1, 3])
def test_ns_step_counts(shape, T):
    run_and_check([shape], torch.bfloat16, dict(HP, ns_steps=T))


@pytest.mark.parametrize("shape", [(24, 1000), (200, 300)], ids=str)
def test_plain_momentum_and_cubic_coefficients(shape):
    run_and_check([shape], torch.bfloat16, dict(HP, nesterov=False))
    run_and_check([shape], torch.float32, dict(HP, coeffs=(1.5, -0.5, 0.0), ns_steps=10))


@pytest.mark.parametrize("shape", [(24, 1000), (24, 10240), (200, 300), (300, 200), (1000, 70)],
                         ids=str)
def test_rms_match_update_scale(shape):
    # s = 0.2 sqrt(max(M, N)) in place of sqrt(max(1, M/N)), both calls
    hp = dict(HP, scale_mode="rms_match")
    run_and_check([shape], torch.bfloat16, hp)
    m = muon()
    W, Gs, M = make_inputs([shape], torch.bfloat16)
    plan = m.Plan([(shape, torch.bfloat16)], scale_mode="rms_match")
    assert abs(plan.groups()[0]["scale"] - 0.2 * max(shape) ** 0.5) < 1e-5
    Wd, Md = [W[0].cuda()], [M[0].cuda()]
    Wb, Mb = [W[0].cuda()], [M[0].cuda()]
    O = gpu_step(plan, Wb, [Gs[0][0].cuda()], Mb, hp)
    gpu_step(plan, Wd, [Gs[0][0].cuda()], Md, hp, ortho=False)
    ref = oracle_step(W, Gs[0], M, hp)
    assert torch.equal(Md[0], Mb[0])
    from helpers import compare_folded
    compare_folded((0, 0), Wd[0].cpu(), W[0], Gs[0][0], M[0], O[0].cpu(), ref[(0, 0)], hp,
                   torch.bfloat16)


@pytest.mark.parametrize("shape", [(24, 1000), (200, 300), (300, 200)], ids=str)
def test_zero_gradient_is_pure_decay(shape):
    m = muon()
    W, Gs, M = make_inputs([shape], torch.bfloat16)
    Wd = [W[0].cuda()]; Gd = [torch.zeros_like(Gs[0][0]).cuda()]; Md = [M[0].cuda()]
    plan = m.Plan([(shape, torch.bfloat16)])
    O = gpu_step(plan, Wd, Gd, Md, HP)
    assert torch.count_nonzero(O[0]).item() == 0 and torch.count_nonzero(Md[0]).item() == 0
    expect = (W[0].float() * np.float32(1 - 0.02 * 0.1)).to(torch.bfloat16)
    assert torch.equal(Wd[0].cpu(), expect)


@pytest.mark.parametrize("shape", [(24, 1000), (200, 300)], ids=str)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_zero_lr_and_wd_leave_params_unchanged(shape, dtype):
    m = muon()
    W, Gs, M = make_inputs([shape], dtype)
    Wd = [W[0].cuda()]
    plan = m.Plan([(shape, dtype)])
    gpu_step(plan, Wd, [Gs[0][0].cuda()], [M[0].cuda()], dict(HP, lr=0.0, wd=0.0))
    assert torch.equal(Wd[0].cpu(), W[0])


@pytest.mark.parametrize("shapes", [[(24, 1000)] * 3, [(200, 300)] * 3], ids=["skinny", "dense"])
def test_slice_results_do_not_depend_on_batch_mates(shapes):
    # RFC section 2: slices are independent; a slice alone and inside a batch
    # must give the same bits
    m = muon()
    W, Gs, M = make_inputs(shapes, torch.bfloat16)
    full = m.Plan([(s, torch.bfloat16) for s in shapes])
    Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
    O = gpu_step(full, Wd, [g.cuda() for g in Gs[0]], Md, HP)
    one = m.Plan([(shapes[1], torch.bfloat16)])
    W1 = [W[1].cuda()]; M1 = [M[1].cuda()]
    O1 = gpu_step(one, W1, [Gs[0][1].cuda()], M1, HP)
    assert torch.equal(O1[0], O[1]) and torch.equal(W1[0], Wd[1]) and torch.equal(M1[0], Md[1])


@pytest.mark.parametrize("shapes", [[(24, 10240)] * 4, [(2, 300, 200)]], ids=["skinny", "dense"])
def test_bitwise_deterministic(shapes):
    m = muon()
    W, Gs, M = make_inputs(shapes, torch.bfloat16)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    outs = []
    for _ in range(2):
        Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
        O = gpu_step(plan, Wd, [g.cuda() for g in Gs[0]], Md, HP)
        outs.append((Wd, Md, O))
    for a, b in zip(outs[0], outs[1]):
        assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_checkpoint_resume_is_bitwise():
    # the caller owns all state: 10 steps == 5 steps, copy out/in, 5 steps
    m = muon()
    shapes = [(24, 1000), (200, 300)]
    W, Gs, M = make_inputs(shapes, torch.bfloat16, steps=10)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    Wa = [w.cuda() for w in W]; Ma = [x.cuda() for x in M]
    for t in range(10):
        gpu_step(plan, Wa, [g.cuda() for g in Gs[t]], Ma, HP, ortho=False)
    Wb = [w.cuda() for w in W]; Mb = [x.cuda() for x in M]
    for t in range(5):
        gpu_step(plan, Wb, [g.cuda() for g in Gs[t]], Mb, HP, ortho=False)
    Wc = [w.cpu().cuda() for w in Wb]; Mc = [x.cpu().cuda() for x in Mb]
    del Wb, Mb
    for t in range(5, 10):
        gpu_step(plan, Wc, [g.cuda() for g in Gs[t]], Mc, HP, ortho=False)
    assert all(torch.equal(a, b) for a, b in zip(Wa, Wc))
    assert all(torch.equal(a, b) for a, b in zip(Ma, Mc))


def test_chunked_workspace_gives_same_bits():
    m = muon()
    shapes = [(5, 200, 150)]
    W, Gs, M = make_inputs(shapes, torch.bfloat16)
    full = m.Plan([(shapes[0], torch.bfloat16)])
    exp_region = 256   # one exponent slot per dense slice, padded to 256 bytes
    per = (full.workspace_bytes - 256 - exp_region) // 5
    capped = m.Plan([(shapes[0], torch.bfloat16)], workspace_cap=256 + 2 * per + exp_region)
    assert capped.groups()[0]["chunk"] == 2
    res = []
    for plan in (full, capped):
        Wd = [W[0].cuda()]; Md = [M[0].cuda()]
        O = gpu_step(plan, Wd, [Gs[0][0].cuda()], Md, HP)
        res.append((Wd[0], Md[0], O[0]))
    assert all(torch.equal(a, b) for a, b in zip(*res))


@pytest.mark.parametrize("ortho", [True, False], ids=["O", "fused"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_first_iterate_scale_prediction_does_not_change_the_bits(dtype, ortho):
    # The dense path writes its first iterate as fp16(V 2^-e) with e predicted
    # from the workspace's previous step of the plan, and rewrites the slices
    # whose prediction missed.  A zeroed workspace (every prediction misses),
    # the same workspace again (every prediction holds) and one filled with
    # random bytes must give the same parameters, momenta and O, bit for bit.
    m = muon()
    shapes = [(3, 200, 150), (300, 200), (130, 260), (2, 256, 640)]
    W, Gs, M = make_inputs(shapes, dtype)
    plan = m.Plan([(s, dtype) for s in shapes])
    ws = m.alloc_workspace(plan)
    gen = torch.Generator(device="cuda").manual_seed(5)
    noise = torch.randint(-128, 128, (plan.workspace_bytes,), dtype=torch.int8, device="cuda",
                          generator=gen).view(torch.uint8)
    res = []
    for k in range(3):
        if k == 2:
            ws.copy_(noise)
            ws[:256].zero_()   # the header's error word must read zero
        Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
        O = gpu_step(plan, Wd, [g.cuda() for g in Gs[0]], Md, HP, ortho=ortho, ws=ws)
        res.append((Wd, Md, O if ortho else []))
    for k in (1, 2):
        for a, b in zip(res[0], res[k]):
            assert all(torch.equal(x, y) for x, y in zip(a, b)), k


@pytest.mark.parametrize("log2_scale", [-12, 40])
def test_dense_path_gradient_scale_extremes(log2_scale):
    # The dense path stores its first iterate as fp16(V 2^-e), e taken from
    # ||V||.  Gradients far from unit scale (std 1e-2 times 2^-12 or 2^40; ||V||
    # stays far above eps) must meet neither fp16 overflow nor a flush to zero:
    # the oracle's O, element-wise parameters and momenta.
    plan = run_and_check([(300, 200), (2, 256, 640)], torch.bfloat16, HP,
                         grad_std=1e-2 * 2.0 ** log2_scale)
    assert all(g["kernel"] == muon().KERNEL_DENSE for g in plan.groups())


def test_skinny_and_dense_paths_agree():
    # the same skinny group through the fused kernel and through the dense
    # GEMM path: both within tolerance of the oracle and of each other
    m = muon()
    shape = (24, 2048)
    W, Gs, M = make_inputs([shape], torch.bfloat16)
    Os = []
    for smax in (64, 0):
        plan = m.Plan([(shape, torch.bfloat16)], skinny_max_m=smax)
        O = gpu_step(plan, [W[0].cuda()], [Gs[0][0].cuda()], [M[0].cuda()], HP)
        Os.append(O[0].cpu().double().numpy())
    assert rel_fro(Os[0], Os[1]) < 2 * TOL["tc16"]


def test_nan_gradient_propagates():
    m = muon()
    for shape in [(24, 512), (200, 300)]:
        W, Gs, M = make_inputs([shape], torch.float32)
        G = Gs[0][0].clone()
        G[3, 7] = float("nan")
        plan = m.Plan([(shape, torch.float32)])
        Wd = [W[0].cuda()]
        gpu_step(plan, Wd, [G.cuda()], [M[0].cuda()], HP, ortho=False)
        assert torch.isnan(Wd[0]).any()


@pytest.mark.parametrize("shape", [(24, 10240), (12, 3000), (16, 520), (32, 2048), (2, 24, 1024),
                                   (200, 300), (300, 200), (2, 200, 150), (1000, 70), (129, 129)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_step_without_O_output(shape, dtype):
    """When O is not requested the update takes other code paths: the fused
    kernel folds -lr s into Q and applies it as one multiply-add, the dense
    path applies it in the epilogue of the last product.  W' must agree with
    the oracle (the O tolerance carried through lr s, plus the rounding of
    W') and with the step that also writes O: on the dense path bit for bit
    (the same fp32 multiply-add of the same accumulator values), on the fused
    kernel within the bf16 rounding of the differently scaled Q.  The
    momentum is the same bits."""
    m = muon()
    W, Gs, M = make_inputs([shape], dtype)
    plan = m.Plan([(shape, dtype)])
    dense = plan.groups()[0]["kernel"] == m.KERNEL_DENSE
    W1, M1 = [W[0].cuda()], [M[0].cuda()]
    O = gpu_step(plan, W1, [Gs[0][0].cuda()], M1, HP)
    W2, M2 = [W[0].cuda()], [M[0].cuda()]
    gpu_step(plan, W2, [Gs[0][0].cuda()], M2, HP, ortho=False)
    assert torch.equal(M1[0], M2[0])
    ref = oracle_step(W, Gs[0], M, HP)
    for e, (Wg1, Wg2, Og) in enumerate(zip(slices(W1[0]), slices(W2[0]), slices(O[0]))):
        Wr, _, Or = ref[(0, e)]
        Mr_, Nr_ = Wr.shape
        lrs = HP["lr"] * float(np.float32(np.sqrt(max(1.0, Mr_ / Nr_))))
        wf = Wg2.double().cpu().numpy()
        wu = Wg1.double().cpu().numpy()
        og = Og.double().cpu().numpy()
        if dtype == torch.bfloat16:
            from helpers import bf16_ulp
            ulp = np.linalg.norm(bf16_ulp(Wr))
        else:
            ulp = np.linalg.norm(np.spacing(np.abs(Wr).astype(np.float32)).astype(np.float64))
        # against the oracle
        assert np.linalg.norm(wf - Wr) <= ulp + lrs * TOL["tc16"] * np.linalg.norm(Or), e
        if dense:
            assert np.array_equal(wf, wu), e
        else:
            # against the step that writes O: bf16 rounding of Q (2^-8 relative
            # per entry, 2^-6 allowed for sums of terms of both signs)
            assert np.linalg.norm(wf - wu) <= ulp + lrs * 2.0 ** -6 * np.linalg.norm(og), e


def test_timed_step_gives_the_same_bits_and_kernel_times():
    # muon_step_timed: the same kernels with an event around each launch
    m = muon()
    shapes = [(24, 1000), (2, 200, 150), (300, 200)]
    W, Gs, M = make_inputs(shapes, torch.bfloat16)
    plan = m.Plan([(s, torch.bfloat16) for s in shapes])
    runs = []
    for timed in (False, True):
        Wd = [w.cuda() for w in W]; Md = [x.cuda() for x in M]
        ws = m.alloc_workspace(plan)
        st = m.PreparedStep(plan, Wd, [g.cuda() for g in Gs[0]], Md, workspace=ws,
                            lr=HP["lr"], beta=HP["beta"], wd=HP["wd"], nesterov=HP["nesterov"],
                            ns_steps=HP["ns_steps"], coeffs=HP["coeffs"])
        t = st.timed() if timed else st()
        torch.cuda.synchronize()
        assert m.workspace_error(ws) == 0
        runs.append((Wd, Md, t))
    assert all(torch.equal(a, b) for a, b in zip(runs[0][0], runs[1][0]))
    assert all(torch.equal(a, b) for a, b in zip(runs[0][1], runs[1][1]))
    t = runs[1][2]
    # one fused launch; per dense group front, finalize + normalize, 3 x 5 products
    assert t["skinny"][1] == 1 and t["front"][1] == 2 and t["norm"][1] == 4
    assert t["gemm"][1] == 30 and t["update"][1] == 0 and t["check"][1] == 0
    assert all(t[k][0] > 0 for k in ("skinny", "front", "norm", "gemm"))
    assert sum(t[k][1] for k in t) == plan.launches(HP["ns_steps"])
