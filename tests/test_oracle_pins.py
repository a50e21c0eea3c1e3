"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes one part of the Muon step (HyperParallel FSDP Muon RFC,
mindspore hyper-parallel issue "HyperParallel FSDP Muon优化器性能优化 RFC")
to something the mathematics decides on its own: closed forms for the
momentum recursion and for rank-one / diagonal / SVD-structured inputs,
the textbook cubic Newton-Schulz polar iteration checked against numpy's
SVD, exact invariants (slice independence, transposition, orthogonal
equivariance), and the update's special cases.  tests/test_oracle_mutants.py
plants typical mistakes in a copy of the oracle and checks that these pins
catch every one.
"""
import json
import os

import numpy as np
import pytest

import oracle

A5 = (3.4445, -4.7750, 2.0315)
EPS = 1e-7
HERE = os.path.dirname(os.path.abspath(__file__))


def p_scalar(x, T, coeffs=A5):
    """Scalar quintic p(x) = a x + b x^3 + c x^5 composed T times."""
    a, b, c = coeffs
    for _ in range(T):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def rand_orth(rng, n, k=None):
    """n x k matrix with orthonormal columns (QR of a Gaussian, numpy)."""
    k = n if k is None else k
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


# ---------------------------------------------------------------- momentum
@pytest.mark.parametrize("nesterov", [False, True])
def test_momentum_constant_gradient_closed_form(nesterov):
    # RFC section 1(1): the iteration's input is the gradient momentum.
    # For a constant G from zero state, M_t = G (1 - beta^t) / (1 - beta).
    rng = np.random.default_rng(3)
    G = rng.standard_normal(257)
    beta = 0.95
    M = np.zeros_like(G)
    for t in range(1, 13):
        M, V = oracle.momentum(G, M, beta, nesterov)
        Mt = G * (1 - beta ** t) / (1 - beta)
        np.testing.assert_allclose(M, Mt, rtol=1e-13, atol=0)
        np.testing.assert_allclose(V, G + beta * Mt if nesterov else Mt, rtol=1e-13, atol=0)


def test_normalize_unit_norm_and_eps():
    rng = np.random.default_rng(4)
    V = rng.standard_normal((5, 9)) * 3.0
    X = oracle.normalize(V)
    r = np.sqrt((V ** 2).sum())
    assert abs(np.sqrt((X ** 2).sum()) - r / (r + EPS)) < 1e-15
    assert np.array_equal(oracle.normalize(np.zeros((3, 4))), np.zeros((3, 4)))


# ---------------------------------------------------------------- Newton-Schulz
@pytest.mark.parametrize("shape", [(1, 37), (37, 1), (1, 1)])
@pytest.mark.parametrize("T", [0, 1, 5])
def test_ns_rank_one_closed_form(shape, T):
    # X = sigma u v^T  =>  A = sigma^2 u u^T and every step maps sigma -> p(sigma)
    rng = np.random.default_rng(5)
    V = rng.standard_normal(shape)
    r = np.sqrt((V ** 2).sum())
    X = oracle.normalize(V)
    O = oracle.newton_schulz(X, T)
    expect = p_scalar(r / (r + EPS), T) * V / r
    np.testing.assert_allclose(O, expect, rtol=1e-13, atol=1e-15)


def test_ns_scalar_reference_values():
    # the scalar composition p^5 at a few points, evaluated through the
    # oracle's matrix iteration on 1x1 inputs
    for x in (1.0, 0.5, 0.25, 0.1, 1 / np.sqrt(24)):
        O = oracle.newton_schulz(np.array([[x]]), 5)
        assert abs(O[0, 0] - p_scalar(x, 5)) < 1e-14


@pytest.mark.parametrize("shape", [(4, 9), (9, 4), (6, 6)])
def test_ns_rectangular_diagonal(shape):
    # a rectangular-diagonal V stays diagonal: O_ii = p^T(d_i / (||d|| + eps))
    d = np.array([0.9, 0.5, 0.3, 0.05, 1.7, 0.2])[: min(shape)]
    V = np.zeros(shape)
    V[np.arange(len(d)), np.arange(len(d))] = d
    O = oracle.newton_schulz(oracle.normalize(V), 5)
    nd = np.sqrt((d ** 2).sum())
    expect = np.zeros(shape)
    expect[np.arange(len(d)), np.arange(len(d))] = p_scalar(d / (nd + EPS), 5)
    np.testing.assert_allclose(O, expect, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("shape", [(7, 19), (19, 7), (12, 12), (1, 5)])
@pytest.mark.parametrize("T", [1, 5])
def test_ns_svd_structured_input(shape, T):
    # V = U diag(s) W^T  =>  O = U diag(p^T(s / (||s|| + eps))) W^T
    rng = np.random.default_rng(6)
    m, n = shape
    k = min(m, n)
    U = rand_orth(rng, m, k)
    W = rand_orth(rng, n, k)
    s = rng.uniform(0.05, 2.0, k)
    V = U @ np.diag(s) @ W.T
    O = oracle.newton_schulz(oracle.normalize(V), T)
    ns = np.sqrt((s ** 2).sum())
    expect = U @ np.diag(p_scalar(s / (ns + EPS), T)) @ W.T
    np.testing.assert_allclose(O, expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", [(6, 15), (15, 6)])
def test_ns_cubic_coefficients_give_polar_factor(shape):
    # textbook cubic Newton-Schulz (a, b, c) = (1.5, -0.5, 0) converges to the
    # polar factor U W^T of V, here obtained from numpy's SVD
    rng = np.random.default_rng(7)
    m, n = shape
    k = min(m, n)
    s = rng.uniform(0.2, 1.0, k)
    V = rand_orth(rng, m, k) @ np.diag(s) @ rand_orth(rng, n, k).T
    O = oracle.newton_schulz(oracle.normalize(V), 40, coeffs=(1.5, -0.5, 0.0))
    u, _, vt = np.linalg.svd(V, full_matrices=False)
    np.testing.assert_allclose(O, u @ vt, rtol=0, atol=1e-12)


def test_ns_transpose_is_exact():
    # working on X^T when M > N makes NS(V^T) = NS(V)^T bit for bit
    rng = np.random.default_rng(8)
    X = oracle.normalize(rng.standard_normal((5, 13)))
    assert np.array_equal(oracle.newton_schulz(X.T.copy(), 5), oracle.newton_schulz(X, 5).T)


def test_ns_orthogonal_equivariance():
    rng = np.random.default_rng(9)
    X = oracle.normalize(rng.standard_normal((8, 21)))
    Q1 = rand_orth(rng, 8)
    Q2 = rand_orth(rng, 21)
    lhs = oracle.newton_schulz(Q1 @ X @ Q2, 5)
    rhs = Q1 @ oracle.newton_schulz(X, 5) @ Q2
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_ns_singular_values_in_range():
    # singular values of O lie in p^5((0, 1]); its max is taken on a fine grid
    grid = np.linspace(1e-6, 1.0, 2_000_001)
    vals = p_scalar(grid, 5)
    i = int(vals.argmax())
    # refine around the grid maximum (p^5 is flat there)
    fine = np.linspace(grid[max(i - 1, 0)], grid[min(i + 1, len(grid) - 1)], 20001)
    pmax = max(vals.max(), p_scalar(fine, 5).max())
    assert 1.2023 < pmax < 1.2024
    rng = np.random.default_rng(10)
    for shape in [(16, 40), (40, 16), (24, 24)]:
        O = oracle.newton_schulz(oracle.normalize(rng.standard_normal(shape)), 5)
        sv = np.linalg.svd(O, compute_uv=False)
        assert sv.max() <= pmax + 1e-12 and sv.min() >= 0


def test_ns_threads_do_not_change_results():
    rng = np.random.default_rng(11)
    X = oracle.normalize(rng.standard_normal((23, 57)))
    assert np.array_equal(oracle.newton_schulz(X, 5, threads=1), oracle.newton_schulz(X, 5, threads=4))


# ---------------------------------------------------------------- update
def test_update_zero_lr_and_wd_keeps_params():
    rng = np.random.default_rng(12)
    W = rng.standard_normal((9, 14)); G = rng.standard_normal((9, 14)); M = rng.standard_normal((9, 14))
    Wn, _, _ = oracle.muon_slice(W, G, M, lr=0.0, beta=0.9, wd=0.0, nesterov=True)
    assert np.array_equal(Wn, W)


def test_update_zero_gradient_is_pure_decay():
    rng = np.random.default_rng(13)
    W = rng.standard_normal((9, 14))
    Z = np.zeros_like(W)
    Wn, Mn, O = oracle.muon_slice(W, Z, Z, lr=0.02, beta=0.95, wd=0.1, nesterov=True)
    assert np.array_equal(O, Z) and np.array_equal(Mn, Z)
    assert np.array_equal(Wn, W * (1 - 0.02 * 0.1))


def test_update_closed_form_and_scale():
    rng = np.random.default_rng(14)
    W = rng.standard_normal((11, 5)); O = rng.standard_normal((11, 5))
    out = oracle.update(W, O, 0.02, 0.1, np.sqrt(11 / 5))
    np.testing.assert_allclose(out, W * (1 - 0.002) - 0.02 * np.sqrt(11 / 5) * O, rtol=1e-15, atol=1e-16)


def test_zero_ns_steps_returns_normalised_momentum():
    rng = np.random.default_rng(15)
    W = rng.standard_normal((6, 10)); G = rng.standard_normal((6, 10)); M = rng.standard_normal((6, 10))
    _, Mn, O = oracle.muon_slice(W, G, M, 0.02, 0.9, 0.1, True, T=0)
    V = G + 0.9 * (0.9 * M + G)
    np.testing.assert_allclose(O, V / (np.sqrt((V ** 2).sum()) + EPS), rtol=1e-14, atol=0)


def test_whole_step_composes_the_pieces():
    rng = np.random.default_rng(16)
    W = rng.standard_normal((12, 7)); G = rng.standard_normal((12, 7)); M = rng.standard_normal((12, 7))
    Wn, Mn, O = oracle.muon_slice(W, G, M, 0.02, 0.95, 0.1, True)
    s = float(np.float32(np.sqrt(12 / 7)))
    m2, v = oracle.momentum(G, M, 0.95, True)
    O2 = oracle.newton_schulz(oracle.normalize(v), 5)
    assert np.array_equal(Mn, m2) and np.array_equal(O, O2)
    assert np.array_equal(Wn, oracle.update(W, O2, 0.02, 0.1, s))


def test_batched_slices_equal_single_slices():
    # RFC section 2: expert slices are independent, so a batch of slices run
    # on several threads equals each slice run alone, bit for bit
    rng = np.random.default_rng(17)
    shapes = [(6, 20), (6, 20), (20, 6), (3, 3), (6, 20)]
    Ws = [rng.standard_normal(s) for s in shapes]
    Gs = [rng.standard_normal(s) for s in shapes]
    Ms = [rng.standard_normal(s) for s in shapes]
    wo, mo, oo, used = oracle.muon_slices(Ws, Gs, Ms, 0.02, 0.95, 0.1, True, threads=3)
    assert used == 3
    for i in range(len(shapes)):
        w1, m1, o1 = oracle.muon_slice(Ws[i], Gs[i], Ms[i], 0.02, 0.95, 0.1, True)
        assert np.array_equal(w1, wo[i]) and np.array_equal(m1, mo[i]) and np.array_equal(o1, oo[i])


# ---------------------------------------------------------------- plan
def _check_plan(shapes, dtypes):
    sg, si, groups = oracle.plan(shapes, dtypes)
    keys = []
    walk = []
    for p, s in enumerate(shapes):
        E, M, N = (s if len(s) == 3 else (1,) + tuple(s))
        walk += [(M, N, dtypes[p])] * E
    assert len(sg) == len(walk)
    # one group per distinct key, numbered by first appearance
    first = {}
    for k in walk:
        first.setdefault(k, len(first))
    assert len(groups) == len(first)
    for s, k in enumerate(walk):
        assert sg[s] == first[k]
    for g, gr in enumerate(groups):
        k = (gr["M"], gr["N"], gr["dtype"])
        assert first[k] == g
        members = [s for s in range(len(walk)) if sg[s] == g]
        assert [si[s] for s in members] == list(range(len(members)))
        assert gr["count"] == len(members)
        assert gr["tr"] == (gr["M"] > gr["N"])
        # nearest float to sqrt(max(1, M/N))
        sc = np.sqrt(max(1.0, gr["M"] / gr["N"]))
        assert gr["scale"] == float(np.float32(sc))
    return sg, si, groups


def test_plan_random_shape_lists():
    rng = np.random.default_rng(18)
    dims = [1, 3, 8, 24, 64]
    for _ in range(50):
        shapes, dtypes = [], []
        for _ in range(rng.integers(1, 12)):
            if rng.random() < 0.4:
                shapes.append((int(rng.integers(1, 5)), int(rng.choice(dims)), int(rng.choice(dims))))
            else:
                shapes.append((int(rng.choice(dims)), int(rng.choice(dims))))
            dtypes.append(str(rng.choice(["bf16", "f32"])))
        _check_plan(shapes, dtypes)


def test_plan_rms_match_scale_gives_update_rms_of_one_fifth():
    # scale_mode "rms_match": s O has RMS 0.2 when O has unit singular values
    # (O O^T = I for M <= N): RMS(O) = sqrt(min(M,N) / (M N)) = 1/sqrt(max(M,N))
    rng = np.random.default_rng(31)
    shapes = [(24, 10240), (64, 64), (300, 70), (70, 300), (4096, 11008), (11008, 4096)]
    _, _, groups = oracle.plan(shapes, ["bf16"] * len(shapes), scale_mode="rms_match")
    assert [(g["M"], g["N"]) for g in groups] == shapes
    for (M, N), g in zip(shapes, groups):
        k = min(M, N)
        if M * N <= 300 * 300:
            Q, _ = np.linalg.qr(rng.standard_normal((max(M, N), k)))
            O = Q.T if M <= N else Q            # unit singular values, shape (M, N)
            rms = np.sqrt(np.mean((g["scale"] * O) ** 2))
        else:
            rms = g["scale"] * np.sqrt(k / (M * N))
        assert abs(rms - 0.2) < 1e-6, (M, N, rms)
    # symmetric in M and N, unlike sqrt(max(1, M/N))
    assert groups[2]["scale"] == groups[3]["scale"] and groups[4]["scale"] == groups[5]["scale"]
    # tabulated: 0.2 sqrt(10240) = 20.238577..., 0.2 sqrt(64) = 1.6
    assert abs(groups[0]["scale"] - 20.2385770) < 1e-5 and groups[1]["scale"] == np.float32(1.6)


def test_plan_rejects_bad_shapes():
    for bad in [[(5,)], [(2, 3, 4, 5)], [(0, 4)], [(3, 0, 2)]]:
        with pytest.raises(ValueError):
            oracle.plan(bad, ["bf16"] * len(bad))


@pytest.mark.parametrize("fixture", sorted(f for f in os.listdir(os.path.join(HERE, "golden"))
                                           if f.startswith("plan_")))
def test_plan_golden(fixture):
    # groupings of the RFC's own workloads, stated in the fixture with its citation
    with open(os.path.join(HERE, "golden", fixture)) as f:
        g = json.load(f)
    shapes = [tuple(s) for s in g["shapes"]]
    sg, si, groups = _check_plan(shapes, [g["dtype"]] * len(shapes))
    got = [[gr["M"], gr["N"], gr["count"], int(gr["tr"])] for gr in groups]
    assert got == g["groups"]


# ---------------------------------------------------------------- loss scaling
def test_all_finite_matches_numpy():
    rng = np.random.default_rng(19)
    G = rng.standard_normal((7, 9))
    assert oracle.all_finite([G, G])
    for bad in (np.inf, -np.inf, np.nan):
        H = G.copy(); H[3, 4] = bad
        assert not oracle.all_finite([G, H]) and not np.isfinite(H).all()


def test_unscale_by_power_of_two_is_exact_and_skips_on_inf():
    rng = np.random.default_rng(20)
    W = rng.standard_normal((6, 11)); G = rng.standard_normal((6, 11)); M = rng.standard_normal((6, 11))
    S = 2.0 ** 12
    wo, mo, oo, found = oracle.muon_slices_amp([W], [G * S], [M], 0.02, 0.95, 0.1, True, 1 / S)
    w1, m1, o1 = oracle.muon_slice(W, G, M, 0.02, 0.95, 0.1, True)
    assert not found
    assert np.array_equal(wo[0], w1) and np.array_equal(mo[0], m1) and np.array_equal(oo[0], o1)
    H = G.copy(); H[0, 0] = np.nan
    wo, mo, oo, found = oracle.muon_slices_amp([W, W], [G, H], [M, M], 0.02, 0.95, 0.1, True, 1 / S)
    assert found and oo is None
    assert all(np.array_equal(x, W) for x in wo) and all(np.array_equal(x, M) for x in mo)


# ---------------------------------------------------------------- AdamW (non-matrix parameters)
def test_adamw_first_step_closed_form():
    # from zero state the bias-corrected moments are g and g^2: the step is
    # lr * g / (|g| + eps) plus the decoupled decay
    rng = np.random.default_rng(22)
    W = rng.standard_normal(301); G = rng.standard_normal(301) * 1e-3
    Z = np.zeros_like(W)
    wo, mo, vo = oracle.adamw(W, G, Z, Z, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1)
    np.testing.assert_allclose(mo, 0.1 * G, rtol=1e-15, atol=0)
    np.testing.assert_allclose(vo, 0.001 * G * G, rtol=1e-12, atol=0)
    np.testing.assert_allclose(wo, W * (1 - 1e-4) - 1e-3 * G / (np.abs(G) + 1e-8), rtol=1e-12, atol=1e-15)


def test_adamw_constant_gradient_keeps_the_first_step():
    # constant g: m_t = g(1-b1^t), v_t = g^2(1-b2^t), so every bias-corrected
    # step equals the first one
    rng = np.random.default_rng(23)
    G = rng.standard_normal(64)
    W = np.zeros(64); M = np.zeros(64); V = np.zeros(64)
    for t in range(1, 8):
        Wn, M, V = oracle.adamw(W, G, M, V, 1e-2, 0.9, 0.99, 1e-12, 0.0, t)
        np.testing.assert_allclose(Wn - W, -1e-2 * np.sign(G), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(M, G * (1 - 0.9 ** t), rtol=1e-12, atol=0)
        W = Wn


def test_adamw_special_cases():
    rng = np.random.default_rng(24)
    W = rng.standard_normal(50); G = rng.standard_normal(50); M = rng.standard_normal(50)
    V = rng.random(50)
    wo, _, _ = oracle.adamw(W, G, M, V, 0.0, 0.9, 0.999, 1e-8, 0.1, 3)
    assert np.array_equal(wo, W)
    Z = np.zeros_like(W)
    wo, mo, vo = oracle.adamw(W, Z, Z, Z, 1e-3, 0.9, 0.999, 1e-8, 0.1, 1)
    assert np.array_equal(wo, W * (1 - 1e-4)) and not mo.any() and not vo.any()
