"""Muon optimizer step on GB300 (sm_103a): Python binding of libmuon_gb300.so.

This module only marshals arguments: it checks torch tensors (device,
dtype, contiguity, shape), takes their device pointers and the current CUDA
stream, and calls the C ABI declared in include/muon_gb300.h.  Every step of
the computation runs in the library's CUDA kernels.  There is no fallback:
if the library is not built, or no sm_103a GPU is current, calls raise.

Entry points mirror the C ABI:
  ns5(G)                         the quintic Newton-Schulz iteration on a stack of matrices
  step(p, g, buf, ...)           one Muon step on a stack of same-shape weights
  step_grouped([(p, g, buf)...]) one Muon step on every group of a model
  adam_step([(p, g, m, v)...])   one DistAdam step on the non-matrix parameters
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "COEFFS", "EPS", "MuonError", "load_library", "library_path", "workspace_bytes",
    "grouped_workspace_bytes", "Workspace", "ns5", "step", "step_noalloc", "step_grouped",
    "GroupedStep", "AdamStep", "adam_step", "ADAM_LR", "ADAM_BETAS", "ADAM_EPS",
    "workspace_status", "noalloc_status", "selftest_wait_timeout", "status_string",
    "kernel_launch_count", "trace_begin", "trace_end",
    "set_fused_ns", "fused_ns", "set_persistent_rounds", "persistent_rounds",
    "set_streamed_apply", "streamed_apply", "KERNEL_KINDS",
]

# Quintic coefficients and rounds as printed in "Muon Custom Sizing 实战", section 2.3.
COEFFS = (3.4445, -4.7750, 2.0315)
STEPS = 5
EPS = 1e-7

# DistAdam settings printed in "Muon Custom Sizing 实战", section 四.
ADAM_LR = 0.008
ADAM_BETAS = (0.8, 0.95)
ADAM_EPS = 1e-8

KERNEL_KINDS = {0: "prologue", 1: "small_ns", 2: "gram", 3: "poly", 4: "update", 5: "apply",
                6: "adam", 7: "fused_ns", 8: "rounds"}
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "timeout",
           5: "workspace"}

_LIB_NAME = "libmuon_gb300.so"
_lib = None


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIB_NAME)


class MuonError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class _Group(ctypes.Structure):
    _fields_ = [("params", ctypes.c_void_p), ("grads", ctypes.c_void_p),
                ("momentum_buf", ctypes.c_void_p), ("g_dtype", ctypes.c_int),
                ("batch", ctypes.c_int), ("rows", ctypes.c_int), ("cols", ctypes.c_int),
                ("lr_scale", ctypes.c_float)]


class _AdamTensor(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("numel", ctypes.c_longlong), ("g_dtype", ctypes.c_int),
                ("lr_scale", ctypes.c_float), ("wd_scale", ctypes.c_float)]


class _TraceRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("round", ctypes.c_int), ("ms", ctypes.c_float),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


def load_library():
    """Load libmuon_gb300.so from this package directory (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -m newton_schulz_step_gb300.build`")
    L = ctypes.CDLL(path)
    vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.muon_workspace_bytes.argtypes = [ci, ci, ci]
    L.muon_workspace_bytes.restype = sz
    L.muon_grouped_workspace_bytes.argtypes = [ctypes.POINTER(_Group), ci]
    L.muon_grouped_workspace_bytes.restype = sz
    L.muon_ns5.argtypes = [vp, ci, vp, ci, ci, ci, ci, cf, cf, cf, cf, vp, sz, vp]
    L.muon_ns5.restype = ci
    L.muon_step.argtypes = [vp, vp, ci, vp, ci, ci, ci, cf, ci, cf, cf, cf, ci, cf, cf, cf, cf,
                            vp, sz, vp]
    L.muon_step.restype = ci
    L.muon_step_noalloc.argtypes = [vp, vp, ci, vp, ci, ci, ci, cf, ci, cf, cf, cf, ci, cf, cf,
                                    cf, cf, vp]
    L.muon_step_noalloc.restype = ci
    L.muon_step_grouped.argtypes = [ctypes.POINTER(_Group), ci, cf, ci, cf, cf, ci, cf, cf, cf,
                                    cf, vp, sz, vp]
    L.muon_step_grouped.restype = ci
    L.muon_workspace_status.argtypes = [vp, sz, vp, ci]
    L.muon_workspace_status.restype = ci
    L.muon_noalloc_status.argtypes = [vp, ci]
    L.muon_noalloc_status.restype = ci
    L.muon_selftest_wait_timeout.argtypes = [vp, sz, ci, vp]
    L.muon_selftest_wait_timeout.restype = ci
    L.muon_adam_step.argtypes = [ctypes.POINTER(_AdamTensor), ci, ci, cf, cf, cf, cf, cf, vp]
    L.muon_adam_step.restype = ci
    L.muon_set_persistent_rounds.argtypes = [ci]
    L.muon_set_persistent_rounds.restype = ci
    L.muon_set_fused_ns.argtypes = [ci]
    L.muon_set_fused_ns.restype = ci
    L.muon_set_streamed_apply.argtypes = [ci]
    L.muon_set_streamed_apply.restype = ci
    L.muon_status_string.argtypes = [ci]
    L.muon_status_string.restype = ctypes.c_char_p
    L.muon_kernel_launch_count.argtypes = []
    L.muon_kernel_launch_count.restype = ctypes.c_ulonglong
    L.muon_trace_begin.argtypes = [ci]
    L.muon_trace_begin.restype = ci
    L.muon_trace_end.argtypes = [ctypes.POINTER(_TraceRecord), ci, ctypes.POINTER(ci)]
    L.muon_trace_end.restype = ci
    _lib = L
    return L


def status_string(code: int) -> str:
    try:
        return load_library().muon_status_string(code).decode()
    except ImportError:
        return _STATUS.get(code, "unknown status")


def _raise(code: int, where: str):
    if code != 0:
        raise MuonError(code, where)


def _gdt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"gradients must be float32 or bfloat16, got {t.dtype}")


def _as3d(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dim() == 2:
        t = t.unsqueeze(0)
    if t.dim() != 3:
        raise ValueError(f"{name} must be [rows, cols] or [batch, rows, cols], got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def workspace_bytes(batch: int, rows: int, cols: int) -> int:
    return int(load_library().muon_workspace_bytes(batch, rows, cols))


def _groups_array(groups):
    arr = (_Group * max(1, len(groups)))()
    for i, (p, g, b, s) in enumerate(groups):
        arr[i].params = p.data_ptr() if p is not None else None
        arr[i].grads = g.data_ptr() if g is not None else None
        arr[i].momentum_buf = b.data_ptr() if b is not None else None
        arr[i].g_dtype = _gdt(g) if g is not None else 1
        arr[i].batch, arr[i].rows, arr[i].cols = (int(x) for x in g.shape)
        arr[i].lr_scale = float(s)
    return arr


def grouped_workspace_bytes(shapes) -> int:
    """shapes: iterable of (batch, rows, cols)."""
    shapes = list(shapes)
    arr = (_Group * max(1, len(shapes)))()
    for i, (b, r, c) in enumerate(shapes):
        arr[i].batch, arr[i].rows, arr[i].cols, arr[i].g_dtype = b, r, c, 1
    return int(load_library().muon_grouped_workspace_bytes(arr, len(shapes)))


class Workspace:
    """Zero-filled device scratch owned by the caller (one per concurrent stream)."""

    def __init__(self, nbytes: int, device=None):
        self.tensor = torch.zeros(max(256, int(nbytes)), dtype=torch.uint8,
                                  device=device if device is not None else "cuda")
        if self.tensor.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.tensor.numel()

    def ensure(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.tensor.device)
        return self


_default_ws = {}


def _workspace(ws, need: int, device) -> Workspace:
    if ws is not None:
        return ws
    key = torch.device(device).index if torch.device(device).index is not None else \
        torch.cuda.current_device()
    w = _default_ws.get(key)
    if w is None:
        w = _default_ws[key] = Workspace(need, device)
    return w.ensure(need)


def ns5(G: torch.Tensor, out: torch.Tensor | None = None, steps: int = STEPS, coeffs=COEFFS,
        eps: float = EPS, workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """The quintic Newton-Schulz iteration of every matrix of G ([b, r, c] or [r, c]); bf16 result."""
    L = load_library()
    squeeze = G.dim() == 2
    G3 = _as3d(G, "G")
    _gdt(G3)
    if out is None:
        out = torch.empty(G3.shape, dtype=torch.bfloat16, device=G3.device)
    out3 = _as3d(out, "out")
    if out3.dtype != torch.bfloat16 or out3.shape != G3.shape:
        raise ValueError("out must be bfloat16 with G's shape")
    b, r, c = G3.shape
    ws = _workspace(workspace, L.muon_workspace_bytes(b, r, c), G3.device)
    a_, b_, c_ = coeffs
    _raise(L.muon_ns5(G3.data_ptr(), _gdt(G3), out3.data_ptr(), b, r, c, steps, a_, b_, c_, eps,
                      ws.ptr, ws.nbytes, _stream_handle(stream)), "muon_ns5")
    return out3[0] if squeeze else out3


def step(params, grads, momentum_buf, *, momentum: float, lr: float, weight_decay: float,
         nesterov: bool = True, lr_scale: float = 0.0, steps: int = STEPS, coeffs=COEFFS,
         eps: float = EPS, workspace: Workspace | None = None, stream=None):
    """One Muon step, in place on params and momentum_buf (fp32, [b, r, c] or [r, c])."""
    L = load_library()
    p3, g3, m3 = _as3d(params, "params"), _as3d(grads, "grads"), _as3d(momentum_buf, "momentum_buf")
    if p3.dtype != torch.float32 or m3.dtype != torch.float32:
        raise TypeError("params and momentum_buf must be float32")
    if not (p3.shape == g3.shape == m3.shape):
        raise ValueError("params, grads and momentum_buf must have the same shape")
    b, r, c = g3.shape
    ws = _workspace(workspace, L.muon_workspace_bytes(b, r, c), g3.device)
    a_, b_, c_ = coeffs
    _raise(L.muon_step(p3.data_ptr(), g3.data_ptr(), _gdt(g3), m3.data_ptr(), b, r, c,
                       momentum, int(bool(nesterov)), lr, weight_decay, lr_scale, steps,
                       a_, b_, c_, eps, ws.ptr, ws.nbytes, _stream_handle(stream)), "muon_step")


def step_noalloc(params, grads, momentum_buf, *, momentum: float, lr: float,
                 weight_decay: float, nesterov: bool = True, lr_scale: float = 0.0,
                 steps: int = STEPS, coeffs=COEFFS, eps: float = EPS, stream=None):
    """step() without a workspace, for callers that may not allocate device memory:
    the library's built-in 64 MiB device scratch (of the tensors' GPU) is used
    instead.  The call runs with the tensors' device current, so the scratch and
    the kernels are on that device."""
    L = load_library()
    p3, g3, m3 = _as3d(params, "params"), _as3d(grads, "grads"), _as3d(momentum_buf, "momentum_buf")
    if p3.dtype != torch.float32 or m3.dtype != torch.float32:
        raise TypeError("params and momentum_buf must be float32")
    if not (p3.shape == g3.shape == m3.shape):
        raise ValueError("params, grads and momentum_buf must have the same shape")
    if not (p3.device == g3.device == m3.device):
        raise ValueError("params, grads and momentum_buf must be on the same device")
    b, r, c = g3.shape
    a_, b_, c_ = coeffs
    with torch.cuda.device(p3.device):
        _raise(L.muon_step_noalloc(p3.data_ptr(), g3.data_ptr(), _gdt(g3), m3.data_ptr(), b, r, c,
                                   momentum, int(bool(nesterov)), lr, weight_decay, lr_scale,
                                   steps, a_, b_, c_, eps, _stream_handle(stream)),
               "muon_step_noalloc")


def _normalise_groups(groups):
    out = []
    for grp in groups:
        if len(grp) == 3:
            p, g, b = grp
            s = 0.0
        else:
            p, g, b, s = grp
        p3, g3, b3 = _as3d(p, "params"), _as3d(g, "grads"), _as3d(b, "momentum_buf")
        if p3.dtype != torch.float32 or b3.dtype != torch.float32:
            raise TypeError("params and momentum_buf must be float32")
        if not (p3.shape == g3.shape == b3.shape):
            raise ValueError("params, grads and momentum_buf must have the same shape")
        _gdt(g3)
        out.append((p3, g3, b3, s))
    return out


class GroupedStep:
    """A prepared muon_step_grouped call: the group table is marshalled once.

    Calling it enqueues one Muon step over every group on the current (or
    given) stream.  The tensors must stay alive and in place between calls.
    """

    def __init__(self, groups, *, momentum: float, lr: float, weight_decay: float,
                 nesterov: bool = True, steps: int = STEPS, coeffs=COEFFS, eps: float = EPS,
                 workspace: Workspace | None = None):
        L = load_library()
        self._groups = _normalise_groups(groups)
        self._arr = _groups_array(self._groups)
        self._n = len(self._groups)
        need = int(L.muon_grouped_workspace_bytes(self._arr, self._n))
        if need == 0 and self._n:
            raise ValueError("invalid group shapes")
        dev = self._groups[0][1].device if self._n else torch.device("cuda")
        self.workspace = workspace.ensure(need) if workspace is not None else Workspace(need, dev)
        self._scalars = (float(momentum), int(bool(nesterov)), float(lr), float(weight_decay),
                         int(steps), *(float(x) for x in coeffs), float(eps))

    def __call__(self, stream=None):
        L = load_library()
        mom, nest, lr, wd, steps, a_, b_, c_, eps = self._scalars
        _raise(L.muon_step_grouped(self._arr, self._n, mom, nest, lr, wd, steps, a_, b_, c_, eps,
                                   self.workspace.ptr, self.workspace.nbytes,
                                   _stream_handle(stream)), "muon_step_grouped")


def step_grouped(groups, *, momentum: float, lr: float, weight_decay: float,
                 nesterov: bool = True, steps: int = STEPS, coeffs=COEFFS, eps: float = EPS,
                 workspace: Workspace | None = None, stream=None):
    """One Muon step over every group: groups = [(params, grads, bufs[, lr_scale]), ...]."""
    GroupedStep(groups, momentum=momentum, lr=lr, weight_decay=weight_decay, nesterov=nesterov,
                steps=steps, coeffs=coeffs, eps=eps, workspace=workspace)(stream)


class AdamStep:
    """A prepared muon_adam_step call over tensors = [(param, grad, exp_avg, exp_avg_sq
    [, lr_scale[, wd_scale]]), ...]; param and the moments are fp32, grad fp32 or bf16,
    all contiguous CUDA tensors of one numel per entry (any shape).  Calling it with
    the step count t (>= 1, after the increment) enqueues one update."""

    def __init__(self, tensors, *, lr: float = ADAM_LR, betas=ADAM_BETAS, eps: float = ADAM_EPS,
                 weight_decay: float = 0.0):
        load_library()
        self._keep = []
        self._arr = (_AdamTensor * max(1, len(tensors)))()
        for i, ent in enumerate(tensors):
            p, g, m, v = ent[:4]
            ls = float(ent[4]) if len(ent) > 4 else 1.0
            ws = float(ent[5]) if len(ent) > 5 else 1.0
            for t, name in ((p, "param"), (g, "grad"), (m, "exp_avg"), (v, "exp_avg_sq")):
                if not t.is_cuda or not t.is_contiguous():
                    raise ValueError(f"{name} must be a contiguous CUDA tensor")
            if p.dtype != torch.float32 or m.dtype != torch.float32 or v.dtype != torch.float32:
                raise TypeError("param, exp_avg and exp_avg_sq must be float32")
            if not (p.numel() == g.numel() == m.numel() == v.numel()):
                raise ValueError("param, grad, exp_avg and exp_avg_sq must have the same numel")
            a = self._arr[i]
            a.param, a.grad, a.exp_avg, a.exp_avg_sq = (t.data_ptr() for t in (p, g, m, v))
            a.numel, a.g_dtype, a.lr_scale, a.wd_scale = p.numel(), _gdt(g), ls, ws
            self._keep.append((p, g, m, v))
        self._n = len(tensors)
        self._scalars = (float(lr), float(betas[0]), float(betas[1]), float(eps),
                         float(weight_decay))

    def __call__(self, step: int, stream=None):
        lr, b1, b2, eps, wd = self._scalars
        _raise(load_library().muon_adam_step(self._arr, self._n, int(step), lr, b1, b2, eps, wd,
                                             _stream_handle(stream)), "muon_adam_step")


def adam_step(tensors, step: int, *, lr: float = ADAM_LR, betas=ADAM_BETAS, eps: float = ADAM_EPS,
              weight_decay: float = 0.0, stream=None):
    """One DistAdam update, in place, of every (param, grad, exp_avg, exp_avg_sq[, lr_scale
    [, wd_scale]]) entry at step count `step` (>= 1)."""
    AdamStep(tensors, lr=lr, betas=betas, eps=eps, weight_decay=weight_decay)(step, stream)


def workspace_status(workspace: Workspace, clear: bool = False, stream=None) -> int:
    """Synchronise and read the workspace's sticky device error word (0 = ok, 4 = timeout)."""
    return int(load_library().muon_workspace_status(workspace.ptr, workspace.nbytes,
                                                    _stream_handle(stream), int(clear)))


def noalloc_status(clear: bool = False, stream=None) -> int:
    """Synchronise and read the error word of step_noalloc()'s built-in scratch on the
    current device (0 = ok, 4 = a bounded wait gave up during the latest call)."""
    return int(load_library().muon_noalloc_status(_stream_handle(stream), int(clear)))


def selftest_wait_timeout(workspace: Workspace | None, limit_us: int = 1000, stream=None):
    """Run the device-side bounded-wait timeout path once (see the C header); with
    workspace None it records the timeout in step_noalloc()'s built-in scratch."""
    ptr, nbytes = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    _raise(load_library().muon_selftest_wait_timeout(ptr, nbytes, limit_us,
                                                     _stream_handle(stream)),
           "muon_selftest_wait_timeout")


def set_fused_ns(enable: bool) -> bool:
    """Run the NS rounds of 64 <= min(r, c) <= 256, max(r, c) <= 512 matrices in one fused
    kernel (True, the default) or in the staged GEMM launches (False); returns the previous
    value."""
    prev = int(load_library().muon_set_fused_ns(int(bool(enable))))
    if prev < 0:
        raise MuonError(1, "muon_set_fused_ns")
    return bool(prev)


def set_persistent_rounds(mode) -> int:
    """Launch structure of the tensor-core NS rounds: True/1 one persistent launch,
    False/0 one launch per stage and round, "auto"/2 (the default) persistent when
    a round is short; returns the previous mode (0, 1 or 2)."""
    m = 2 if mode == "auto" else int(mode)
    prev = int(load_library().muon_set_persistent_rounds(m))
    if prev < 0:
        raise MuonError(1, "muon_set_persistent_rounds")
    return prev


class persistent_rounds:
    """Context manager: `with persistent_rounds(True): ...` runs the block with the
    persistent rounds kernel."""

    def __init__(self, mode):
        self.mode = mode
        self.prev = None

    def __enter__(self):
        self.prev = set_persistent_rounds(self.mode)
        return self

    def __exit__(self, *exc):
        set_persistent_rounds(self.prev)
        return False


def set_streamed_apply(enable: bool) -> bool:
    """Run the parameter write beside the persistent rounds kernel's last round (True,
    the default, where the call allows it) or after it (False); returns the previous
    value."""
    return bool(load_library().muon_set_streamed_apply(int(bool(enable))))


class streamed_apply:
    """Context manager: `with streamed_apply(False): ...` runs the block with the
    parameter write after the rounds kernel."""

    def __init__(self, enable: bool):
        self.enable = enable
        self.prev = None

    def __enter__(self):
        self.prev = set_streamed_apply(self.enable)
        return self

    def __exit__(self, *exc):
        set_streamed_apply(self.prev)
        return False


class fused_ns:
    """Context manager: `with fused_ns(False): ...` runs the block on the staged path."""

    def __init__(self, enable: bool):
        self.enable = bool(enable)
        self.prev = None

    def __enter__(self):
        self.prev = set_fused_ns(self.enable)
        return self

    def __exit__(self, *exc):
        set_fused_ns(self.prev)
        return False


def kernel_launch_count() -> int:
    return int(load_library().muon_kernel_launch_count())


def trace_begin(max_launches: int = 4096):
    _raise(load_library().muon_trace_begin(max_launches), "muon_trace_begin")


def trace_end(max_records: int = 4096):
    """Stop tracing; list of {kind, round, ms, flops, bytes} in launch order."""
    recs = (_TraceRecord * max(1, max_records))()
    n = ctypes.c_int(0)
    _raise(load_library().muon_trace_end(recs, max_records, ctypes.byref(n)), "muon_trace_end")
    return [{"kind": KERNEL_KINDS.get(r.kind, str(r.kind)), "round": r.round, "ms": r.ms,
             "flops": r.flops, "bytes": r.bytes} for r in recs[: n.value]]
