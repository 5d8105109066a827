"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, plans workspaces, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest
import torch

import newton_schulz_step_gb300 as muon

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon_gb300.h")

OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT, WORKSPACE = range(6)
A, B, C = muon.COEFFS


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(muon.library_path()):
        from newton_schulz_step_gb300 import build
        build.build()
    return muon.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    raw = ctypes.CDLL(muon.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for code in range(6):
        s = muon.status_string(code)
        assert isinstance(s, str) and s
    assert muon.status_string(99) == "unknown status"


def _align(x):
    return (x + 255) // 256 * 256


def test_workspace_bytes(lib):
    assert lib.muon_workspace_bytes(0, 5, 7) == 256
    assert lib.muon_workspace_bytes(-1, 5, 7) == 0
    assert lib.muon_workspace_bytes(1, 0, 7) == 0
    assert lib.muon_workspace_bytes(1, 70000, 7) == 0
    # small path: fp32 m x n per matrix
    assert lib.muon_workspace_bytes(3, 12, 768) == 256 + _align(3 * 12 * 768 * 4)
    # tensor-core path: one completion counter per matrix (u32, after the status
    # block), then X0, X1 (m x ldx bf16), A, B (m x lda bf16), norm partials
    b, r, c = 2, 300, 130          # tall: m = 130, n = 300
    m, n, ldx, lda = 130, 300, 304, 136
    parts = 4                      # ceil(15 prologue tiles / 4)
    buffers = 2 * _align(b * m * ldx * 2) + 2 * _align(b * m * lda * 2) + _align(b * parts * 4)
    assert lib.muon_workspace_bytes(b, r, c) == 256 + _align(b * 4) + buffers
    # the grouped size is the sum of the per-group regions (counters only for
    # tensor-core matrices)
    grp = muon.grouped_workspace_bytes([(3, 12, 768), (2, 300, 130)])
    assert grp == 256 + _align(2 * 4) + _align(3 * 12 * 768 * 4) + buffers
    grp = muon.grouped_workspace_bytes([(70, 64, 64), (2, 300, 130)])
    assert grp == 256 + _align(72 * 4) + (
        2 * _align(70 * 64 * 64 * 2) + 2 * _align(70 * 64 * 64 * 2) + _align(70 * 1 * 4)) + buffers


def test_trace_without_launches(lib):
    muon.trace_begin(16)
    assert muon.trace_end() == []


def _step(lib, **kw):
    args = dict(params=0x1000, grads=0x2000, gdt=1, buf=0x3000, batch=1, rows=64, cols=64,
                mom=0.95, nest=1, lr=0.02, wd=0.01, scale=0.0, steps=5, a=A, b=B, c=C, eps=1e-7,
                ws=0x10000, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.muon_step(args["params"], args["grads"], args["gdt"], args["buf"], args["batch"],
                         args["rows"], args["cols"], args["mom"], args["nest"], args["lr"],
                         args["wd"], args["scale"], args["steps"], args["a"], args["b"],
                         args["c"], args["eps"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(params=None), INVALID), (dict(grads=None), INVALID), (dict(buf=None), INVALID),
    (dict(params=0x1004), INVALID), (dict(grads=0x2002), INVALID),
    (dict(batch=-1), INVALID), (dict(rows=0), INVALID), (dict(cols=70000), INVALID),
    (dict(gdt=7), INVALID), (dict(steps=0), INVALID), (dict(steps=17), INVALID),
    (dict(mom=1.5), INVALID), (dict(mom=float("nan")), INVALID), (dict(eps=-1.0), INVALID),
    (dict(a=float("inf")), INVALID), (dict(lr=float("nan")), INVALID),
    (dict(ws=None), WORKSPACE), (dict(ws=0x10010), WORKSPACE), (dict(wsb=1024), WORKSPACE),
    (dict(batch=0), OK),
])
def test_step_argument_errors_before_any_launch(lib, kw, code):
    assert _step(lib, **kw) == code


def test_grouped_argument_errors(lib):
    assert lib.muon_step_grouped(None, 0, 0.95, 1, 0.02, 0.01, 5, A, B, C, 1e-7, None, 0, None) \
        == WORKSPACE
    assert lib.muon_step_grouped(None, 2, 0.95, 1, 0.02, 0.01, 5, A, B, C, 1e-7, 0x10000, 1 << 20,
                                 None) == INVALID
    arr = (muon._Group * 1)()
    arr[0].batch, arr[0].rows, arr[0].cols, arr[0].g_dtype = 1, 64, 64, 1
    arr[0].params, arr[0].grads, arr[0].momentum_buf = 0x1000, None, 0x3000
    assert lib.muon_step_grouped(arr, 1, 0.95, 1, 0.02, 0.01, 5, A, B, C, 1e-7, 0x10000, 1 << 30,
                                 None) == INVALID
    assert lib.muon_grouped_workspace_bytes(None, -1) == 0


def test_ns5_argument_errors(lib):
    f = lib.muon_ns5
    assert f(0x1000, 1, None, 1, 64, 64, 5, A, B, C, 1e-7, 0x10000, 1 << 30, None) == INVALID
    assert f(None, 1, 0x2000, 1, 64, 64, 5, A, B, C, 1e-7, 0x10000, 1 << 30, None) == INVALID
    assert f(0x1000, 1, 0x2000, 1, 64, 64, 99, A, B, C, 1e-7, 0x10000, 1 << 30, None) == INVALID
    assert f(0x1000, 1, 0x2000, 0, 64, 64, 5, A, B, C, 1e-7, 0x10000, 1 << 30, None) == OK


def test_selftest_argument_errors(lib):
    assert lib.muon_selftest_wait_timeout(0x10010, 1024, 1000, None) == WORKSPACE
    assert lib.muon_selftest_wait_timeout(0x10000, 16, 1000, None) == WORKSPACE
    assert lib.muon_selftest_wait_timeout(0x10000, 1024, 0, None) == INVALID
    assert lib.muon_selftest_wait_timeout(0x10000, 1024, 200000, None) == INVALID
    assert lib.muon_selftest_wait_timeout(None, 0, 0, None) == INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_noalloc_scratch_calls_without_gpu_are_refused(lib):
    # NULL workspace = the built-in scratch of muon_step_noalloc: without a device
    # there is no scratch, and nothing is launched
    assert lib.muon_selftest_wait_timeout(None, 0, 1000, None) in (UNSUPPORTED, CUDA)
    assert lib.muon_noalloc_status(None, 0) in (UNSUPPORTED, CUDA)


def test_workspace_status_argument_errors(lib):
    assert lib.muon_workspace_status(None, 1024, None, 0) == WORKSPACE
    assert lib.muon_workspace_status(0x10010, 1024, None, 0) == WORKSPACE
    assert lib.muon_workspace_status(0x10000, 16, None, 0) == WORKSPACE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_well_formed_call_without_gpu_is_refused(lib):
    # no device: the call must refuse (never fall back to the CPU); pointers are never touched
    code = _step(lib)
    assert code in (UNSUPPORTED, CUDA)
    with pytest.raises(Exception):
        muon.ns5(torch.zeros(4, 64, 64))   # CPU tensor: the binding refuses as well


def _adam_arr(n=1, numel=1000, ptr=0x10000, dtype=1):
    arr = (muon._AdamTensor * max(1, n))()
    for i in range(n):
        a = arr[i]
        a.param, a.grad, a.exp_avg, a.exp_avg_sq = ptr, ptr + 0x100000, ptr + 0x200000, ptr + 0x300000
        a.numel, a.g_dtype, a.lr_scale, a.wd_scale = numel, dtype, 1.0, 1.0
    return arr


def test_adam_argument_errors(lib):
    f = lib.muon_adam_step
    arr = _adam_arr()
    assert f(arr, -1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    assert f(None, 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    assert f(arr, 1, 0, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID        # step counts from 1
    assert f(arr, 1, 1, 0.008, 1.0, 0.95, 1e-8, 0.0, None) == INVALID        # beta1 < 1
    assert f(arr, 1, 1, 0.008, 0.8, -0.1, 1e-8, 0.0, None) == INVALID        # beta2 >= 0
    assert f(arr, 1, 1, 0.008, 0.8, 0.95, -1e-8, 0.0, None) == INVALID       # eps >= 0
    assert f(arr, 1, 1, float("nan"), 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    assert f(arr, 1, 1, 0.008, 0.8, 0.95, 1e-8, float("inf"), None) == INVALID
    assert f(_adam_arr(ptr=0x10008), 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    assert f(_adam_arr(dtype=7), 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    assert f(_adam_arr(numel=-5), 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    bad = _adam_arr()
    bad[0].grad = None
    assert f(bad, 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    bad = _adam_arr()
    bad[0].lr_scale = -1.0
    assert f(bad, 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == INVALID
    # nothing to do is OK without touching a device
    assert f(None, 0, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == OK
    empty = _adam_arr(numel=0)
    empty[0].param = empty[0].grad = empty[0].exp_avg = empty[0].exp_avg_sq = None
    assert f(empty, 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU refusal")
def test_adam_without_gpu_is_refused(lib):
    code = lib.muon_adam_step(_adam_arr(), 1, 1, 0.008, 0.8, 0.95, 1e-8, 0.0, None)
    assert code in (UNSUPPORTED, CUDA)
