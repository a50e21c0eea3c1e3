"""Python handle on the fp64 CPU oracle of the Muon step (muon_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product package.  It shares no
code with the CUDA path.  Inputs are converted to float64 numpy arrays (bf16
and fp32 values convert exactly); outputs are float64.

Every function follows the HyperParallel FSDP Muon RFC (mindspore
hyper-parallel issue "HyperParallel FSDP Muon优化器性能优化 RFC"); the
readings of the steps it leaves open are stated in muon_oracle.cpp.

Parity pinned by tests/test_oracle_pins.py (closed forms, invariants,
textbook special cases); no function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "muon_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-7
DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)

# dtype codes used by the plan key; any distinct integers work for the oracle
DTYPE_CODES = {"bf16": 0, "f32": 1}

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_ip = ctypes.POINTER(ctypes.c_int)
_fp = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (IEEE double, no FMA contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + ".tmp%d" % os.getpid()
            subprocess.check_call([
                "g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp])
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB_PATH lets the mutation test load a deliberately broken
        # copy of the oracle in a child process; it is never set otherwise.
        path = os.environ.get("ORACLE_LIB_PATH")
        if not path:
            path = build()
        L = ctypes.CDLL(path)
        L.oracle_plan.restype = ctypes.c_int
        L.oracle_plan.argtypes = [ctypes.c_int, _ip, _i64p, _ip, _ip, _ip, ctypes.c_int,
                                  _i64p, _i64p, _ip, _ip, _ip, _fp, ctypes.c_int]
        L.oracle_momentum.argtypes = [ctypes.c_int64, _dp, _dp, ctypes.c_double, ctypes.c_int, _dp, _dp]
        L.oracle_normalize.argtypes = [ctypes.c_int64, _dp, ctypes.c_double, _dp]
        L.oracle_newton_schulz.argtypes = [ctypes.c_int64, ctypes.c_int64, _dp, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                           ctypes.c_int, _dp]
        L.oracle_update.argtypes = [ctypes.c_int64, _dp, _dp, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, _dp]
        L.oracle_muon_slice.argtypes = [ctypes.c_int64, ctypes.c_int64, _dp, _dp, _dp,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_int, ctypes.c_int, _dp, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
        L.oracle_all_finite.restype = ctypes.c_int
        L.oracle_all_finite.argtypes = [ctypes.c_int64, _dp]
        L.oracle_unscale.argtypes = [ctypes.c_int64, _dp, ctypes.c_double, _dp]
        L.oracle_adamw.argtypes = [ctypes.c_int64, _dp, _dp, _dp, _dp, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
        PP = ctypes.POINTER(_dp)
        L.oracle_muon_slices.restype = ctypes.c_int
        L.oracle_muon_slices.argtypes = [ctypes.c_int, _i64p, _i64p, PP, PP, PP,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                         ctypes.c_int, ctypes.c_int, _dp, ctypes.c_double,
                                         _dp, ctypes.c_int, PP, PP, PP]
        _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    """float64 C-contiguous copy of a numpy array or CPU torch tensor."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


# --------------------------------------------------------------------------
# plan
SCALE_MODES = {"sqrt_ratio": 0, "rms_match": 1}


def plan(shapes: Sequence[Tuple[int, ...]], dtypes: Sequence[str], scale_mode: str = "sqrt_ratio"):
    """Group slices by (M, N, dtype) in order of first appearance.

    Returns (slice_group, slice_index, groups) with groups a list of dicts
    {M, N, dtype, count, tr, scale(float32)}; scale_mode "sqrt_ratio" gives
    s = sqrt(max(1, M/N)), "rms_match" s = 0.2 sqrt(max(M, N))."""
    n = len(shapes)
    ndim = (ctypes.c_int * max(n, 1))()
    dims = (ctypes.c_int64 * max(3 * n, 1))()
    dt = (ctypes.c_int * max(n, 1))()
    total = 0
    for p, s in enumerate(shapes):
        ndim[p] = len(s)
        for k, d in enumerate(s[:3]):
            dims[3 * p + k] = d
        dt[p] = DTYPE_CODES[dtypes[p]]
        total += s[0] if len(s) == 3 else 1
    sg = (ctypes.c_int * max(total, 1))()
    si = (ctypes.c_int * max(total, 1))()
    cap = max(n, 1)
    gM = (ctypes.c_int64 * cap)(); gN = (ctypes.c_int64 * cap)()
    gd = (ctypes.c_int * cap)(); gc = (ctypes.c_int * cap)(); gt = (ctypes.c_int * cap)()
    gs = (ctypes.c_float * cap)()
    r = lib().oracle_plan(n, ndim, dims, dt, sg, si, cap, gM, gN, gd, gc, gt, gs,
                          SCALE_MODES[scale_mode])
    if r < 0:
        raise ValueError("oracle_plan rejected the shapes (code %d)" % r)
    inv = {v: k for k, v in DTYPE_CODES.items()}
    groups = [dict(M=gM[g], N=gN[g], dtype=inv[gd[g]], count=gc[g], tr=bool(gt[g]),
                   scale=float(np.float32(gs[g]))) for g in range(r)]
    return list(sg[:total]), list(si[:total]), groups


# --------------------------------------------------------------------------
# per-step pieces
def momentum(G, Mom, beta: float, nesterov: bool):
    g = _f64(G); m = _f64(Mom)
    mo = np.empty_like(g); v = np.empty_like(g)
    lib().oracle_momentum(g.size, _ptr(g), _ptr(m), beta, int(nesterov), _ptr(mo), _ptr(v))
    return mo, v


def normalize(V, eps: float = EPS):
    v = _f64(V); x = np.empty_like(v)
    lib().oracle_normalize(v.size, _ptr(v), eps, _ptr(x))
    return x


def newton_schulz(X, T: int = 5, coeffs=DEFAULT_COEFFS, threads: int = 1):
    x = _f64(X)
    assert x.ndim == 2
    o = np.empty_like(x)
    lib().oracle_newton_schulz(x.shape[0], x.shape[1], _ptr(x), T, coeffs[0], coeffs[1],
                               coeffs[2], threads, _ptr(o))
    return o


def update(W, O, lr: float, wd: float, scale: float):
    w = _f64(W); o = _f64(O); out = np.empty_like(w)
    lib().oracle_update(w.size, _ptr(w), _ptr(o), lr, wd, scale, _ptr(out))
    return out


def muon_slice(W, G, Mom, lr, beta, wd, nesterov, T=5, coeffs=DEFAULT_COEFFS,
               eps=EPS, scale=None, threads: int = 1):
    """One [M, N] slice through the whole step.  Returns (W', M', O) in fp64."""
    w = _f64(W); g = _f64(G); m = _f64(Mom)
    M, N = w.shape
    if scale is None:
        scale = float(np.float32(np.sqrt(max(1.0, M / N))))
    wo = np.empty_like(w); mo = np.empty_like(w); o = np.empty_like(w)
    c = np.asarray(coeffs, dtype=np.float64)
    lib().oracle_muon_slice(M, N, _ptr(w), _ptr(g), _ptr(m), lr, beta, wd, int(nesterov), T,
                            _ptr(c), eps, scale, threads, _ptr(wo), _ptr(mo), _ptr(o))
    return wo, mo, o


def muon_slices(Ws: List, Gs: List, Moms: List, lr, beta, wd, nesterov, T=5,
                coeffs=DEFAULT_COEFFS, eps=EPS, scales: Optional[List[float]] = None,
                threads: int = 1, want_O: bool = True):
    """Independent [M, N] slices spread over `threads` host threads.

    Returns (W's, M's, Os or None, threads used)."""
    n = len(Ws)
    w = [_f64(x) for x in Ws]; g = [_f64(x) for x in Gs]; m = [_f64(x) for x in Moms]
    Ms = (ctypes.c_int64 * n)(*[x.shape[0] for x in w])
    Ns = (ctypes.c_int64 * n)(*[x.shape[1] for x in w])
    if scales is None:
        scales = [float(np.float32(np.sqrt(max(1.0, x.shape[0] / x.shape[1])))) for x in w]
    sc = np.asarray(scales, dtype=np.float64)
    wo = [np.empty_like(x) for x in w]; mo = [np.empty_like(x) for x in w]
    oo = [np.empty_like(x) for x in w] if want_O else None
    PA = _dp * n
    c = np.asarray(coeffs, dtype=np.float64)
    used = lib().oracle_muon_slices(
        n, Ms, Ns, PA(*[_ptr(x) for x in w]), PA(*[_ptr(x) for x in g]),
        PA(*[_ptr(x) for x in m]), lr, beta, wd, int(nesterov), T, _ptr(c), eps, _ptr(sc),
        threads, PA(*[_ptr(x) for x in wo]), PA(*[_ptr(x) for x in mo]),
        PA(*[_ptr(x) for x in oo]) if want_O else None)
    return wo, mo, oo, used


def all_finite(Gs) -> bool:
    """True when every value of every gradient is finite (loss-scaler check)."""
    return all(lib().oracle_all_finite(g.size, _ptr(g)) == 1 for g in (_f64(x) for x in Gs))


def unscale(G, inv_scale: float):
    g = _f64(G); out = np.empty_like(g)
    lib().oracle_unscale(g.size, _ptr(g), inv_scale, _ptr(out))
    return out


def muon_slices_amp(Ws, Gs, Moms, lr, beta, wd, nesterov, inv_scale: float, **kw):
    """The loss-scaled step: if any gradient value of any slice is inf or NaN
    the step is skipped (found_inf = True, every W and M unchanged);
    otherwise the step runs on G * inv_scale.  Returns (W's, M's, Os, found_inf)."""
    if not all_finite(Gs):
        return [_f64(w) for w in Ws], [_f64(m) for m in Moms], None, True
    wo, mo, oo, _ = muon_slices(Ws, [unscale(g, inv_scale) for g in Gs], Moms, lr, beta, wd,
                                nesterov, **kw)
    return wo, mo, oo, False


def adamw(W, G, M, V, lr, beta1, beta2, eps, wd, step: int):
    """AdamW step (bias-corrected, decoupled decay) for one tensor of any
    shape.  Returns (W', M', V') in fp64."""
    w = _f64(W); g = _f64(G); m = _f64(M); v = _f64(V)
    wo = np.empty_like(w); mo = np.empty_like(w); vo = np.empty_like(w)
    lib().oracle_adamw(w.size, _ptr(w), _ptr(g), _ptr(m), _ptr(v), lr, beta1, beta2, eps, wd,
                       step, _ptr(wo), _ptr(mo), _ptr(vo))
    return wo, mo, vo


def param_slices(t) -> List:
    """The [M, N] slices of a 2D or 3D parameter (2D is a one-slice stack)."""
    if t.dim() == 2:
        return [t]
    return [t[e] for e in range(t.shape[0])]


# --------------------------------------------------------------------------
# assignment of slices to replicas (several GPUs)
#
# HyperParallel FSDP Muon RFC, section 4 (HSDP grouped computation): every
# replica group holds all parameters, each orthogonalises only the ones a
# greedy algorithm assigns to it for an even compute load, and the updated
# parameters are then broadcast; section 2: the E slices of an [E, M, N]
# expert tensor are mathematically independent, so a slice is the unit.
# Readings (the RFC names the algorithm "greedy" and the goal "balanced
# compute", nothing more):
#   * the load of a slice is its time on the roofline of one GPU,
#     max(Newton-Schulz flops / tensor rate, optimizer-state bytes / HBM rate),
#     flops in the standard count T (4 m^2 n + 2 m^3) (X X^T and B X at
#     2 m^2 n each, A A at 2 m^3 per step), bytes 3 es + 8 per element
#     (G read, W read and written in the parameter dtype; fp32 momentum read
#     and written);
#   * greedy = longest first: slices in decreasing load (equal loads: lower
#     global slice id first), each to the replica with the least load so far
#     (equal: the lower rank).
def slice_costs(shapes: Sequence[Tuple[int, ...]], dtypes: Sequence[str], ns_steps: int,
                flops_per_s: float, bytes_per_s: float) -> List[float]:
    """Load (seconds) of every slice, in global slice order."""
    costs = []
    for shape, dt in zip(shapes, dtypes):
        E, M, N = (1, shape[0], shape[1]) if len(shape) == 2 else tuple(shape)
        m, n = min(M, N), max(M, N)
        es = 2 if dt == "bf16" else 4
        flops = ns_steps * (4 * m * m * n + 2 * m * m * m)     # exact Python integers
        nbytes = m * n * (3 * es + 8)
        cost = max(flops / flops_per_s, nbytes / bytes_per_s)
        costs.extend([cost] * E)
    return costs


def partition(costs: Sequence[float], world: int) -> Tuple[List[int], List[float]]:
    """Greedy longest-first assignment of slices to `world` replicas.

    Returns (owner of each slice, summed load of each replica)."""
    order = sorted(range(len(costs)), key=lambda s: (-costs[s], s))
    load = [0.0] * world
    owner = [0] * len(costs)
    for s in order:
        r = min(range(world), key=lambda k: (load[k], k))
        owner[s] = r
        load[r] += costs[s]
    return owner, load
