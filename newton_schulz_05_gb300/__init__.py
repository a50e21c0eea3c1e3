"""Muon optimizer step on one GB300: thin Python binding of libmuon.

Every step of the optimizer runs in libmuon's CUDA kernels (C ABI declared in
include/muon.h); this module only marshals tensor pointers and the stream.
PyTorch provides device memory and streams.  There is no CPU fallback: if
libmuon.so is missing or cannot be loaded, importing the binding raises.

The step (HyperParallel FSDP Muon RFC, mindspore hyper-parallel issue
"HyperParallel FSDP Muon优化器性能优化 RFC", sections 1-3 and 6):
momentum / Nesterov -> per-slice Frobenius normalisation -> quintic
Newton-Schulz on min(M,N) x max(M,N) -> W' = W (1 - lr wd) - lr s O, with
slices of equal trailing dims grouped into one batch.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmuon.so")

MUON_OK = 0
MUON_BF16, MUON_F32 = 0, 1
MODE_TC16, MODE_FP32 = 0, 1
KERNEL_SKINNY, KERNEL_DENSE = 0, 1
DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)

_DTYPES = {torch.bfloat16: MUON_BF16, torch.float32: MUON_F32}
_MODES = {"tc16": MODE_TC16, "fp32": MODE_FP32}
# update scale s of a [M, N] slice (MUON_SCALE_* in include/muon.h)
SCALE_MODES = {"sqrt_ratio": 0, "rms_match": 1}


class MuonError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


class _Shape(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int), ("dims", ctypes.c_int64 * 3), ("dtype", ctypes.c_int)]


class _Options(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("eps", ctypes.c_float),
                ("workspace_cap", ctypes.c_size_t), ("skinny_max_m", ctypes.c_int),
                ("scale_mode", ctypes.c_int)]


class _GroupInfo(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("m", ctypes.c_int64),
                ("n", ctypes.c_int64), ("dtype", ctypes.c_int), ("count", ctypes.c_int),
                ("tr", ctypes.c_int), ("scale", ctypes.c_float), ("kernel", ctypes.c_int),
                ("cluster", ctypes.c_int), ("chunk", ctypes.c_int)]


KERNEL_CLASSES = ("skinny", "front", "norm", "gemm", "update", "check")   # MUON_KC_*


class _KernelTimes(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_float * len(KERNEL_CLASSES)),
                ("launches", ctypes.c_int * len(KERNEL_CLASSES))]


EXPORTS = ["muon_options_default", "muon_plan", "muon_plan_workspace_bytes",
           "muon_plan_num_groups", "muon_plan_num_slices", "muon_plan_group",
           "muon_plan_slice", "muon_step", "muon_step_ortho", "muon_workspace_error",
           "muon_plan_launches", "muon_plan_destroy", "muon_status_string", "muon_step_static",
           "muon_step_amp", "muon_adamw_step", "muon_plan_partition", "muon_static_error",
           "muon_step_timed", "muon_step_host", "muon_plan_host_unit_bytes",
           "muon_host_alloc", "muon_host_free"]

STATIC_WORKSPACE_BYTES = 32 << 20   # MUON_STATIC_WORKSPACE_BYTES in include/muon.h

# default rates of the slice loads of Plan.partition: dense fp16/bf16 tensor
# throughput and STREAM-copy HBM bandwidth of one GB300, as measured (only
# their ratio matters to the assignment)
GB300_FLOPS = 1.88e15
GB300_HBM_BYTES = 6.78e12

_lib = None


def load(path: str = LIB_PATH):
    """Load libmuon.so (built by newton_schulz_05_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libmuon.so not built at %s: run newton_schulz_05_gb300.build.build() "
                           "(there is no CPU fallback)" % path)
    L = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    PP = ctypes.POINTER(ctypes.c_void_p)
    L.muon_options_default.argtypes = [ctypes.POINTER(_Options)]
    L.muon_options_default.restype = None
    L.muon_plan.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, ctypes.POINTER(_Options), PP]
    L.muon_plan_workspace_bytes.argtypes = [vp, ctypes.POINTER(sz)]
    L.muon_plan_num_groups.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    L.muon_plan_num_slices.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    L.muon_plan_group.argtypes = [vp, ctypes.c_int, ctypes.POINTER(_GroupInfo)]
    L.muon_plan_slice.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                  ctypes.POINTER(ctypes.c_int)]
    step_args = [vp, PP, PP, PP, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_int,
                 ctypes.c_int, ctypes.POINTER(ctypes.c_float), vp, sz, vp]
    L.muon_step.argtypes = step_args
    L.muon_step_ortho.argtypes = step_args + [PP]
    L.muon_step_timed.argtypes = step_args + [ctypes.POINTER(_KernelTimes)]
    L.muon_step_host.argtypes = step_args[:12] + [vp, sz, sz, vp]
    L.muon_plan_host_unit_bytes.argtypes = [vp, ctypes.POINTER(sz)]
    L.muon_host_alloc.argtypes = [sz, PP]
    L.muon_host_free.argtypes = [vp]
    L.muon_step_static.argtypes = step_args[:10] + [vp]
    L.muon_step_amp.argtypes = step_args[:10] + [ctypes.c_float, vp, vp, sz, vp]
    L.muon_adamw_step.argtypes = [ctypes.c_int, PP, PP, PP, PP, ctypes.POINTER(ctypes.c_int64),
                                  ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  ctypes.c_float, ctypes.c_float, ctypes.c_int, vp]
    L.muon_workspace_error.argtypes = [vp, vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    L.muon_static_error.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    L.muon_plan_launches.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    L.muon_plan_partition.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_double, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_double)]
    L.muon_plan_destroy.argtypes = [vp]
    L.muon_plan_destroy.restype = None
    L.muon_status_string.argtypes = [ctypes.c_int]
    L.muon_status_string.restype = ctypes.c_char_p
    for fn in ("muon_plan", "muon_plan_workspace_bytes", "muon_plan_num_groups",
               "muon_plan_num_slices", "muon_plan_group", "muon_plan_slice", "muon_step",
               "muon_step_ortho", "muon_workspace_error", "muon_plan_launches",
               "muon_step_static", "muon_step_amp", "muon_adamw_step", "muon_plan_partition",
               "muon_static_error", "muon_step_timed", "muon_step_host",
               "muon_plan_host_unit_bytes", "muon_host_alloc", "muon_host_free"):
        getattr(L, fn).restype = ctypes.c_int
    _lib = L
    return L


def status_string(s: int) -> str:
    return load().muon_status_string(s).decode()


def _check(status: int, what: str):
    if status != MUON_OK:
        raise MuonError(status, what)


def _shape_of(t) -> Tuple[Tuple[int, ...], int]:
    if isinstance(t, torch.Tensor):
        if t.dtype not in _DTYPES:
            raise TypeError("parameters must be bf16 or fp32, got %s" % t.dtype)
        return tuple(t.shape), _DTYPES[t.dtype]
    shape, dtype = t
    return tuple(shape), _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)


class Plan:
    """Host-side grouping of parameters by trailing dims (muon_plan)."""

    def __init__(self, params: Sequence, mode: str = "tc16", eps: float = 1e-7,
                 workspace_cap: int = 0, skinny_max_m: int = 64,
                 scale_mode: str = "sqrt_ratio"):
        L = load()
        specs = [_shape_of(p) for p in params]
        n = len(specs)
        arr = (_Shape * max(n, 1))()
        for i, (shape, dt) in enumerate(specs):
            arr[i].ndim = len(shape)
            for k in range(min(len(shape), 3)):
                arr[i].dims[k] = shape[k]
            arr[i].dtype = dt
        opt = _Options()
        L.muon_options_default(ctypes.byref(opt))
        opt.mode = _MODES[mode]
        opt.eps = eps
        opt.workspace_cap = workspace_cap
        opt.skinny_max_m = skinny_max_m
        opt.scale_mode = SCALE_MODES[scale_mode]
        h = ctypes.c_void_p()
        _check(L.muon_plan(arr, n, ctypes.byref(opt), ctypes.byref(h)), "muon_plan")
        self._h = h
        self.shapes = [s for s, _ in specs]
        self.dtypes = [d for _, d in specs]
        self.mode = mode

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.muon_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    @property
    def workspace_bytes(self) -> int:
        v = ctypes.c_size_t()
        _check(load().muon_plan_workspace_bytes(self._h, ctypes.byref(v)), "workspace_bytes")
        return v.value

    @property
    def num_slices(self) -> int:
        v = ctypes.c_int()
        _check(load().muon_plan_num_slices(self._h, ctypes.byref(v)), "num_slices")
        return v.value

    def groups(self) -> List[dict]:
        L = load()
        n = ctypes.c_int()
        _check(L.muon_plan_num_groups(self._h, ctypes.byref(n)), "num_groups")
        out = []
        for g in range(n.value):
            gi = _GroupInfo()
            _check(L.muon_plan_group(self._h, g, ctypes.byref(gi)), "plan_group")
            out.append({f: getattr(gi, f) for f, _ in _GroupInfo._fields_})
        return out

    def slice(self, param: int, e: int) -> Tuple[int, int]:
        g, i = ctypes.c_int(), ctypes.c_int()
        _check(load().muon_plan_slice(self._h, param, e, ctypes.byref(g), ctypes.byref(i)),
               "plan_slice")
        return g.value, i.value

    @property
    def host_unit_bytes(self) -> int:
        """Smallest staging unit of muon_step_host for this plan."""
        v = ctypes.c_size_t()
        _check(load().muon_plan_host_unit_bytes(self._h, ctypes.byref(v)), "host_unit_bytes")
        return v.value

    def launches(self, ns_steps: int = 5) -> int:
        v = ctypes.c_int()
        _check(load().muon_plan_launches(self._h, ns_steps, ctypes.byref(v)), "plan_launches")
        return v.value

    def partition(self, world: int, ns_steps: int = 5, flops_per_s: float = GB300_FLOPS,
                  bytes_per_s: float = GB300_HBM_BYTES) -> Tuple[List[int], List[float]]:
        """muon_plan_partition: owner rank of every global slice and the summed
        load (seconds) of every rank."""
        ns = self.num_slices
        owner = (ctypes.c_int * max(ns, 1))()
        loads = (ctypes.c_double * max(world, 1))()
        _check(load().muon_plan_partition(self._h, world, ns_steps, flops_per_s, bytes_per_s,
                                          owner, loads), "plan_partition")
        return list(owner[:ns]), list(loads[:world])


def _ptrs(ts) -> ctypes.Array:
    return (ctypes.c_void_p * max(len(ts), 1))(*[t.data_ptr() for t in ts])


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def step(plan: Plan, params, grads, momentum, *, lr: float, beta: float, wd: float,
         nesterov: bool = True, ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
         workspace: torch.Tensor, stream=None, ortho=None) -> None:
    """Enqueue one Muon step (muon_step / muon_step_ortho) on `stream`.

    params / grads / momentum: lists of contiguous CUDA tensors in plan order;
    momentum is fp32.  ortho (optional): fp32 tensors shaped like params that
    receive the orthogonalised momentum O."""
    L = load()
    n = len(plan.shapes)
    if not (len(params) == len(grads) == len(momentum) == n):
        raise ValueError("expected %d params, grads and momentum tensors" % n)
    for i, (p, g, m) in enumerate(zip(params, grads, momentum)):
        if tuple(p.shape) != plan.shapes[i] or tuple(g.shape) != plan.shapes[i] or \
                tuple(m.shape) != plan.shapes[i]:
            raise ValueError("tensor %d does not match the plan's shape %s" % (i, plan.shapes[i]))
        if _DTYPES.get(p.dtype) != plan.dtypes[i] or g.dtype != p.dtype or m.dtype != torch.float32:
            raise TypeError("tensor %d: dtype mismatch with the plan" % i)
        if not (p.is_cuda and g.is_cuda and m.is_cuda):
            raise ValueError("tensor %d is not on a CUDA device" % i)
        if not (p.is_contiguous() and g.is_contiguous() and m.is_contiguous()):
            raise ValueError("tensor %d is not contiguous" % i)
    c = (ctypes.c_float * 3)(*coeffs)
    args = [plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum), lr, beta, wd,
            int(bool(nesterov)), ns_steps, c, ctypes.c_void_p(workspace.data_ptr()),
            workspace.numel() * workspace.element_size(), ctypes.c_void_p(_stream_handle(stream))]
    if ortho is None:
        _check(L.muon_step(*args), "muon_step")
    else:
        for i, o in enumerate(ortho):
            if tuple(o.shape) != plan.shapes[i] or o.dtype != torch.float32 or not o.is_contiguous():
                raise ValueError("ortho %d must be a contiguous fp32 tensor of the param's shape" % i)
        _check(L.muon_step_ortho(*args, _ptrs(ortho)), "muon_step_ortho")


def step_static(plan: Plan, params, grads, momentum, *, lr: float, beta: float, wd: float,
                nesterov: bool = True, ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
                stream=None) -> None:
    """muon_step_static: one step with the library's static device scratch
    instead of a caller-allocated workspace (for callers that cannot
    allocate; plans needing more than STATIC_WORKSPACE_BYTES are rejected).
    Calls that overlap on the GPU share, and race on, that scratch."""
    c = (ctypes.c_float * 3)(*coeffs)
    _check(load().muon_step_static(plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum), lr,
                                   beta, wd, int(bool(nesterov)), ns_steps, c,
                                   ctypes.c_void_p(_stream_handle(stream))), "muon_step_static")


def static_error(stream=None, clear: bool = True) -> int:
    """Device error word that the last step_static on the current device left
    in the library's static scratch (synchronises the stream); 0 when every
    device-side wait of that step completed."""
    code = ctypes.c_int()
    _check(load().muon_static_error(ctypes.c_void_p(_stream_handle(stream)), int(clear),
                                    ctypes.byref(code)), "static_error")
    return code.value


def step_amp(plan: Plan, params, grads, momentum, *, lr: float, beta: float, wd: float,
             inv_scale: float, found_inf: torch.Tensor, nesterov: bool = True, ns_steps: int = 5,
             coeffs=DEFAULT_COEFFS, workspace: torch.Tensor, stream=None) -> None:
    """muon_step_amp: one step on loss-scaled gradients (grads * inv_scale),
    skipped entirely when any gradient value is inf or NaN; found_inf is a
    one-element int32 CUDA tensor that receives 1 (skipped) or 0."""
    if found_inf.dtype != torch.int32 or not found_inf.is_cuda or found_inf.numel() < 1:
        raise ValueError("found_inf must be a CUDA int32 tensor")
    c = (ctypes.c_float * 3)(*coeffs)
    _check(load().muon_step_amp(plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum), lr,
                                beta, wd, int(bool(nesterov)), ns_steps, c, inv_scale,
                                ctypes.c_void_p(found_inf.data_ptr()),
                                ctypes.c_void_p(workspace.data_ptr()),
                                workspace.numel() * workspace.element_size(),
                                ctypes.c_void_p(_stream_handle(stream))), "muon_step_amp")


def adamw_step(params, grads, exp_avg, exp_avg_sq, *, lr: float, beta1: float = 0.9,
               beta2: float = 0.999, eps: float = 1e-8, wd: float = 0.0, step: int,
               stream=None) -> None:
    """muon_adamw_step: one AdamW step over every tensor (one launch per 256
    tensors).  params/grads: contiguous CUDA tensors of one dtype (bf16 or
    fp32); exp_avg/exp_avg_sq: fp32 tensors of the same sizes."""
    n = len(params)
    if not (len(grads) == len(exp_avg) == len(exp_avg_sq) == n):
        raise ValueError("expected equally many params, grads and moment tensors")
    dt = {torch.bfloat16: MUON_BF16, torch.float32: MUON_F32}.get(params[0].dtype if n else torch.float32)
    if dt is None:
        raise TypeError("parameters must be bf16 or fp32")
    for p, g, m, v in zip(params, grads, exp_avg, exp_avg_sq):
        if p.dtype != params[0].dtype or g.dtype != p.dtype or m.dtype != torch.float32 or \
                v.dtype != torch.float32:
            raise TypeError("dtype mismatch")
        if not (p.numel() == g.numel() == m.numel() == v.numel()):
            raise ValueError("size mismatch")
        if not all(t.is_cuda and t.is_contiguous() for t in (p, g, m, v)):
            raise ValueError("tensors must be contiguous CUDA tensors")
    numel = (ctypes.c_int64 * max(n, 1))(*[p.numel() for p in params])
    _check(load().muon_adamw_step(n, _ptrs(params), _ptrs(grads), _ptrs(exp_avg), _ptrs(exp_avg_sq),
                                  numel, dt, lr, beta1, beta2, eps, wd, step,
                                  ctypes.c_void_p(_stream_handle(stream))), "muon_adamw_step")


def workspace_error(workspace: torch.Tensor, stream=None, clear: bool = True) -> int:
    """Device error word of the workspace (synchronises the stream)."""
    code = ctypes.c_int()
    _check(load().muon_workspace_error(ctypes.c_void_p(workspace.data_ptr()),
                                       ctypes.c_void_p(_stream_handle(stream)), int(clear),
                                       ctypes.byref(code)), "workspace_error")
    return code.value


def _host_free(addr: int) -> None:
    load().muon_host_free(ctypes.c_void_p(addr))


def alloc_host(numel: int, dtype: torch.dtype) -> torch.Tensor:
    """A CPU tensor of `numel` elements in page-locked, huge-page-backed host
    memory from muon_host_alloc, for the state muon_step_host streams (zeros).
    The memory is released by muon_host_free once the tensor and every view
    of it are gone."""
    import weakref
    es = torch.empty(0, dtype=dtype).element_size()
    nbytes = int(numel) * es
    if nbytes <= 0:
        raise ValueError("alloc_host needs at least one element")
    p = ctypes.c_void_p()
    _check(load().muon_host_alloc(ctypes.c_size_t(nbytes), ctypes.byref(p)), "muon_host_alloc")
    buf = (ctypes.c_uint8 * nbytes).from_address(p.value)
    weakref.finalize(buf, _host_free, p.value)   # runs when the last tensor view dies
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype)


def alloc_workspace(plan: Plan, device=None) -> torch.Tensor:
    """A zeroed device workspace of the plan's size (torch's allocator returns
    256-byte aligned blocks)."""
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=device or "cuda")
    if ws.data_ptr() % 256:
        raise RuntimeError("workspace not 256-byte aligned")
    return ws


class Muon:
    """Muon optimizer over a fixed list of parameter tensors.

    Holds the plan, the fp32 momentum buffers and the workspace; ``step(grads)``
    runs one optimizer step in place on the CUDA stream."""

    def __init__(self, params: Sequence[torch.Tensor], lr: float = 0.02, beta: float = 0.95,
                 wd: float = 0.1, nesterov: bool = True, ns_steps: int = 5,
                 coeffs=DEFAULT_COEFFS, mode: str = "tc16", eps: float = 1e-7):
        self.params = list(params)
        self.plan = Plan(self.params, mode=mode, eps=eps)
        self.momentum = [torch.zeros_like(p, dtype=torch.float32) for p in self.params]
        self.workspace = alloc_workspace(self.plan, self.params[0].device if self.params else None)
        self.hp = dict(lr=lr, beta=beta, wd=wd, nesterov=nesterov, ns_steps=ns_steps,
                       coeffs=coeffs)

    def step(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        step(self.plan, self.params, grads, self.momentum, workspace=self.workspace,
             stream=stream, **self.hp)


class PreparedStep:
    """A muon_step call with its argument arrays marshalled once.

    For a fixed set of tensors (the usual case: parameters, gradient buffers
    and momentum never move) calling the object enqueues one step with a
    single C call and no per-call Python-side validation."""

    def __init__(self, plan: Plan, params, grads, momentum, *, lr: float, beta: float, wd: float,
                 nesterov: bool = True, ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
                 workspace: torch.Tensor, stream=None, ortho=None):
        # validate once through the checked path's rules
        n = len(plan.shapes)
        if not (len(params) == len(grads) == len(momentum) == n):
            raise ValueError("expected %d params, grads and momentum tensors" % n)
        for i, (p, g, m) in enumerate(zip(params, grads, momentum)):
            if tuple(p.shape) != plan.shapes[i] or g.shape != p.shape or m.shape != p.shape:
                raise ValueError("tensor %d does not match the plan's shape" % i)
            if _DTYPES.get(p.dtype) != plan.dtypes[i] or g.dtype != p.dtype or m.dtype != torch.float32:
                raise TypeError("tensor %d: dtype mismatch with the plan" % i)
            if not (p.is_cuda and g.is_cuda and m.is_cuda and p.is_contiguous() and
                    g.is_contiguous() and m.is_contiguous()):
                raise ValueError("tensor %d must be a contiguous CUDA tensor" % i)
        self._keep = (plan, list(params), list(grads), list(momentum), workspace, ortho)
        self._fn = load().muon_step_ortho if ortho is not None else load().muon_step
        c = (ctypes.c_float * 3)(*coeffs)
        self._args = [plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum),
                      ctypes.c_float(lr), ctypes.c_float(beta), ctypes.c_float(wd),
                      ctypes.c_int(int(bool(nesterov))), ctypes.c_int(ns_steps), c,
                      ctypes.c_void_p(workspace.data_ptr()),
                      ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                      ctypes.c_void_p(_stream_handle(stream))]
        if ortho is not None:
            self._args.append(_ptrs(ortho))

    def __call__(self) -> None:
        _check(self._fn(*self._args), "muon_step")

    def timed(self) -> dict:
        """The same step through muon_step_timed (not with O outputs): a CUDA
        event before every launch; synchronises the stream and returns
        {kernel class: (device ms, launches)}."""
        if len(self._args) != 13:
            raise ValueError("timed steps do not write O")
        t = _KernelTimes()
        _check(load().muon_step_timed(*self._args, ctypes.byref(t)), "muon_step_timed")
        return {k: (t.ms[i], t.launches[i]) for i, k in enumerate(KERNEL_CLASSES)}


class PreparedHostStep:
    """A muon_step_host call (parameters, gradients and momenta in host
    memory, streamed through a device staging buffer) with its argument
    arrays marshalled once.  params/grads/momentum: CPU tensors, contiguous
    (page-locked for full copy bandwidth: alloc_host gives memory that keeps
    it when the state is cold); the call updates params and
    momentum in place once the stream has run it.  The staging is cut into
    units of unit_bytes (default: a third of it)."""

    def __init__(self, plan: Plan, params, grads, momentum, *, lr: float, beta: float, wd: float,
                 nesterov: bool = True, ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
                 workspace: torch.Tensor, staging: torch.Tensor, unit_bytes: int = 0,
                 stream=None):
        n = len(plan.shapes)
        if not (len(params) == len(grads) == len(momentum) == n):
            raise ValueError("expected %d params, grads and momentum tensors" % n)
        for i, (p, g, m) in enumerate(zip(params, grads, momentum)):
            if tuple(p.shape) != plan.shapes[i] or g.shape != p.shape or m.shape != p.shape:
                raise ValueError("tensor %d does not match the plan's shape" % i)
            if _DTYPES.get(p.dtype) != plan.dtypes[i] or g.dtype != p.dtype or m.dtype != torch.float32:
                raise TypeError("tensor %d: dtype mismatch with the plan" % i)
            if p.is_cuda or g.is_cuda or m.is_cuda or not (p.is_contiguous() and g.is_contiguous()
                                                          and m.is_contiguous()):
                raise ValueError("tensor %d must be a contiguous host tensor" % i)
        if not staging.is_cuda or staging.data_ptr() % 256:
            raise ValueError("staging must be a 256-byte aligned CUDA buffer")
        self._keep = (plan, list(params), list(grads), list(momentum), workspace, staging)
        c = (ctypes.c_float * 3)(*coeffs)
        self._args = [plan.handle, _ptrs(params), _ptrs(grads), _ptrs(momentum),
                      ctypes.c_float(lr), ctypes.c_float(beta), ctypes.c_float(wd),
                      ctypes.c_int(int(bool(nesterov))), ctypes.c_int(ns_steps), c,
                      ctypes.c_void_p(workspace.data_ptr()),
                      ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                      ctypes.c_void_p(staging.data_ptr()),
                      ctypes.c_size_t(staging.numel() * staging.element_size()),
                      ctypes.c_size_t(unit_bytes or staging.numel() * staging.element_size() // 3),
                      ctypes.c_void_p(_stream_handle(stream))]

    def __call__(self) -> None:
        _check(load().muon_step_host(*self._args), "muon_step_host")


class Partition:
    """Slices of a set of parameters dealt to `world` replicas that all hold
    every parameter (HyperParallel FSDP Muon RFC, section 4: each replica
    orthogonalises the parameters a greedy algorithm assigns to it, then the
    updated parameters are broadcast; section 2: a slice of an [E, M, N]
    tensor is the unit).  Owners come from muon_plan_partition, so every
    replica computes the same assignment without communicating.

    ``broadcast`` sends each rank's updated slices to the others through
    torch.distributed (one broadcast per owner and dtype of a packed buffer);
    it moves bytes only."""

    def __init__(self, plan: Plan, world: int, ns_steps: int = 5,
                 flops_per_s: float = GB300_FLOPS, bytes_per_s: float = GB300_HBM_BYTES):
        self.world = world
        self.owner, self.rank_load = plan.partition(world, ns_steps, flops_per_s, bytes_per_s)
        # global slice id -> (param, e)
        self.slice_keys = []
        for p, shape in enumerate(plan.shapes):
            for e in range(shape[0] if len(shape) == 3 else 1):
                self.slice_keys.append((p, e))
        self._bufs = {}

    def owned(self, rank: int) -> List[Tuple[int, int]]:
        """(param, slice) pairs of `rank`, in global slice order."""
        return [k for k, o in zip(self.slice_keys, self.owner) if o == rank]

    @staticmethod
    def view(t: torch.Tensor, key: Tuple[int, int]) -> torch.Tensor:
        """The 2-D [M, N] slice `key` = (param, e) of the list's tensor."""
        return t if t.dim() == 2 else t[key[1]]

    def views(self, tensors: Sequence[torch.Tensor], rank: int) -> List[torch.Tensor]:
        return [self.view(tensors[p], (p, e)) for p, e in self.owned(rank)]

    def broadcast(self, params: Sequence[torch.Tensor], group=None) -> None:
        """Every rank's slices of `params` sent from that rank to all others."""
        import torch.distributed as dist
        if self.world == 1:
            return
        me = dist.get_rank(group) if group is not None else dist.get_rank()
        for r in range(self.world):
            vs = self.views(params, r)
            by_dtype = {}
            for v in vs:
                by_dtype.setdefault(v.dtype, []).append(v)
            for dt, lst in by_dtype.items():
                total = sum(v.numel() for v in lst)
                key = (r, dt, lst[0].device)
                buf = self._bufs.get(key)
                if buf is None or buf.numel() != total:
                    buf = torch.empty(total, dtype=dt, device=lst[0].device)
                    self._bufs[key] = buf
                if me == r:
                    torch.cat([v.reshape(-1) for v in lst], out=buf)
                src = dist.get_global_rank(group, r) if group is not None else r
                dist.broadcast(buf, src=src, group=group)
                if me != r:
                    off = 0
                    for v in lst:
                        v.copy_(buf[off:off + v.numel()].view_as(v))
                        off += v.numel()


class ShardedMuon:
    """Muon over the replicas of a process group: every rank holds all
    parameters and the full (already reduced) gradients, orthogonalises and
    updates only the slices the Partition gives it, keeps fp32 momentum for
    those slices only, then the updated slices are broadcast from their
    owners.  The update on each rank runs in libmuon's kernels over a plan of
    the rank's own 2-D slice views; the result equals the single-replica step
    slice for slice (every slice is computed independently of the others)."""

    def __init__(self, params: Sequence[torch.Tensor], rank: int, world: int, group=None,
                 lr: float = 0.02, beta: float = 0.95, wd: float = 0.1, nesterov: bool = True,
                 ns_steps: int = 5, coeffs=DEFAULT_COEFFS, mode: str = "tc16", eps: float = 1e-7,
                 flops_per_s: float = GB300_FLOPS, bytes_per_s: float = GB300_HBM_BYTES):
        self.params = list(params)
        self.rank, self.world, self.group = rank, world, group
        self.partition = Partition(Plan(self.params, mode=mode, eps=eps), world, ns_steps,
                                   flops_per_s, bytes_per_s)
        self.owned = self.partition.owned(rank)
        self.param_views = self.partition.views(self.params, rank)
        self.plan = Plan(self.param_views, mode=mode, eps=eps)
        self.momentum = [torch.zeros(v.shape, dtype=torch.float32, device=v.device)
                         for v in self.param_views]
        dev = self.params[0].device if self.params else None
        self.workspace = alloc_workspace(self.plan, dev)
        self.hp = dict(lr=lr, beta=beta, wd=wd, nesterov=nesterov, ns_steps=ns_steps,
                       coeffs=coeffs)

    def update_owned(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        """The step on this rank's slices only (no communication)."""
        if self.param_views:
            step(self.plan, self.param_views, self.partition.views(grads, self.rank),
                 self.momentum, workspace=self.workspace, stream=stream, **self.hp)

    def step(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        self.update_owned(grads, stream)
        if self.world > 1:
            self.partition.broadcast(self.params, self.group)


class MuonWithAdamW:
    """Muon for the matrix parameters (2-D matrices and 3-D [E, M, N] stacks)
    and AdamW for the others (1-D biases and norm scales): the split of the
    Paddle Muon sharding PR ("Support Muon sharding optimizer comm overlap"),
    which keeps 2-D and 1-D gradients in separate buffers because the two
    kinds of parameter take different update rules.

    ``step(grads)`` takes the gradients in the order of ``params`` and runs
    one muon_step over the matrix parameters and one muon_adamw_step per
    dtype over the others, all on the stream."""

    def __init__(self, params: Sequence[torch.Tensor], lr: float = 0.02, beta: float = 0.95,
                 wd: float = 0.1, nesterov: bool = True, ns_steps: int = 5,
                 coeffs=DEFAULT_COEFFS, mode: str = "tc16", eps: float = 1e-7,
                 adamw_lr: float = 3e-4, betas=(0.9, 0.999), adamw_eps: float = 1e-8,
                 adamw_wd: float = 0.0):
        self.params = list(params)
        self.matrix_idx, self.other_idx, self.groups = self.route(self.params)
        mats = [self.params[i] for i in self.matrix_idx]
        self.muon = Muon(mats, lr=lr, beta=beta, wd=wd, nesterov=nesterov, ns_steps=ns_steps,
                         coeffs=coeffs, mode=mode, eps=eps) if mats else None
        self.exp_avg = {i: torch.zeros(self.params[i].numel(), dtype=torch.float32,
                                       device=self.params[i].device) for i in self.other_idx}
        self.exp_avg_sq = {i: torch.zeros_like(self.exp_avg[i]) for i in self.other_idx}
        self.adamw = dict(lr=adamw_lr, beta1=betas[0], beta2=betas[1], eps=adamw_eps, wd=adamw_wd)
        self.t = 0

    @staticmethod
    def route(params: Sequence[torch.Tensor]):
        """(indices of the Muon parameters, indices of the AdamW parameters,
        {dtype: AdamW indices}) for a parameter list."""
        matrix = [i for i, p in enumerate(params) if p.dim() in (2, 3)]
        other = [i for i, p in enumerate(params) if p.dim() not in (2, 3)]
        groups = {}
        for i in other:
            groups.setdefault(params[i].dtype, []).append(i)
        return matrix, other, groups

    def step(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        if len(grads) != len(self.params):
            raise ValueError("expected one gradient per parameter")
        self.t += 1
        if self.muon is not None:
            self.muon.step([grads[i] for i in self.matrix_idx], stream=stream)
        for _, idx in self.groups.items():
            adamw_step([self.params[i].view(-1) for i in idx], [grads[i].reshape(-1) for i in idx],
                       [self.exp_avg[i] for i in idx], [self.exp_avg_sq[i] for i in idx],
                       step=self.t, stream=stream, **self.adamw)
