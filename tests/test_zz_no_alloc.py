"""muon_step_noalloc (through the C ABI) against muon_step and the oracle.

muon_step_noalloc serves callers that cannot allocate device memory (an
allocator that owns the whole GPU, a plug-in limited to the memory it is given,
a loop that forbids allocation after start-up): its scratch is an array built
into the library instead of a caller workspace.  It runs the same kernels on
the same inputs, so its results must be bit-identical to muon_step's; they are
also checked against the CPU float64 oracle.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import newton_schulz_step_gb300 as muon
import oracle

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2    # bf16 tensor-core NS, as in the parity tests
SMALL_TOL = 1e-4  # fp32 small-matrix NS
EW_TOL = 1e-5    # fp32 elementwise momentum buffer
SCRATCH = 64 << 20
TIMEOUT = 4      # MUON_ERR_TIMEOUT
A_, B_, C_ = muon.COEFFS


def _rel(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def _f64(t):
    return t.detach().float().cpu().double().numpy()


def _noalloc(L, p, g, b, stream):
    gdt = 1 if g.dtype == torch.bfloat16 else 0
    return L.muon_step_noalloc(p.data_ptr(), g.data_ptr(), gdt, b.data_ptr(), *g.shape, 0.95, 1,
                               0.02, 0.01, 0.0, 5, A_, B_, C_, 1e-7, stream)


def _check_against_oracle(p_before, g, b_before, p, b):
    shape = tuple(g.shape)
    tol = SMALL_TOL if min(shape[1:]) < 64 else NS_TOL
    for i in range(shape[0]):
        p_ref, b_ref, _ = oracle.muon_step(_f64(p_before[i]), _f64(g[i]), _f64(b_before[i]),
                                           momentum=0.95, lr=0.02, weight_decay=0.01)
        assert _rel(_f64(b[i]), b_ref) < EW_TOL
        base = 0.9998 * _f64(p_before[i])
        assert _rel(_f64(p[i]) - base, p_ref - base) < tol


@pytest.mark.parametrize("shape,gdt", [((4, 768, 3072), torch.bfloat16),
                                       ((3, 520, 300), torch.float32),
                                       ((2, 160, 288), torch.bfloat16),
                                       ((10, 12, 768), torch.bfloat16)])
def test_noalloc_matches_workspace_entry_on_two_calls(shape, gdt):
    L = muon.load_library()
    assert L.muon_workspace_bytes(*shape) <= SCRATCH
    gen = torch.Generator().manual_seed(123)
    p0 = (0.02 * torch.randn(*shape, generator=gen)).cuda()
    b0 = (1e-3 * torch.randn(*shape, generator=gen)).cuda()
    grads = [(1e-3 * torch.randn(*shape, generator=gen)).to(gdt).cuda() for _ in range(2)]
    p_ref, b_ref = p0.clone(), b0.clone()
    p_new, b_new = p0.clone(), b0.clone()
    ws = muon.Workspace(L.muon_workspace_bytes(*shape))
    stream = torch.cuda.current_stream().cuda_stream
    gdt_code = 1 if gdt == torch.bfloat16 else 0
    for g in grads:                       # two calls in a row, state carried over
        p_before, b_before = p_new.clone(), b_new.clone()
        code = L.muon_step(p_ref.data_ptr(), g.data_ptr(), gdt_code, b_ref.data_ptr(), *shape,
                           0.95, 1, 0.02, 0.01, 0.0, 5, A_, B_, C_, 1e-7, ws.ptr, ws.nbytes,
                           stream)
        assert code == 0, muon.status_string(code)
        code = _noalloc(L, p_new, g, b_new, stream)
        assert code == 0, muon.status_string(code)
        torch.cuda.synchronize()
        assert muon.noalloc_status() == 0
        # the same kernels on the same inputs: bit-identical to muon_step
        assert torch.equal(b_new, b_ref)
        assert torch.equal(p_new, p_ref)
        _check_against_oracle(p_before, g, b_before, p_new, b_new)


def test_noalloc_status_reports_a_timeout_and_the_next_call_starts_clean():
    # a bounded wait that runs out on the built-in scratch (NULL workspace) is
    # reported by muon_noalloc_status; the next noalloc call clears the word
    # before its kernels run, computes a correct step, and reports success
    L = muon.load_library()
    shape = (2, 256, 640)
    gen = torch.Generator().manual_seed(7)
    p = (0.02 * torch.randn(*shape, generator=gen)).cuda()
    b = (1e-3 * torch.randn(*shape, generator=gen)).cuda()
    g = (1e-3 * torch.randn(*shape, generator=gen)).to(torch.bfloat16).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert _noalloc(L, p.clone(), g, b.clone(), stream) == 0   # first call: address lookup
    torch.cuda.synchronize()
    assert muon.noalloc_status() == 0
    muon.selftest_wait_timeout(None, limit_us=1000)
    assert muon.noalloc_status() == TIMEOUT
    assert muon.noalloc_status() == TIMEOUT                     # sticky until cleared
    p_before, b_before = p.clone(), b.clone()
    assert _noalloc(L, p, g, b, stream) == 0
    torch.cuda.synchronize()
    assert muon.noalloc_status() == 0
    _check_against_oracle(p_before, g, b_before, p, b)
    # and a word cleared by the query itself stays clear
    muon.selftest_wait_timeout(None, limit_us=1000)
    assert muon.noalloc_status(clear=True) == TIMEOUT
    assert muon.noalloc_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = muon.load_library()
    shape = (1, 4096, 4096)                # needs ~134 MB of scratch
    assert L.muon_workspace_bytes(*shape) > SCRATCH
    # rejected before anything is enqueued: the pointers are never touched
    code = L.muon_step_noalloc(0x1000, 0x2000, 1, 0x3000, *shape, 0.95, 1, 0.02, 0.01, 0.0, 5,
                               A_, B_, C_, 1e-7, None)
    assert code == 5   # MUON_ERR_WORKSPACE


def test_noalloc_binding_runs_on_the_tensors_device():
    # the binding makes the tensors' device current for the call
    shape = (1, 128, 256)
    gen = torch.Generator().manual_seed(9)
    p0 = 0.02 * torch.randn(*shape, generator=gen)
    b0 = 1e-3 * torch.randn(*shape, generator=gen)
    g = (1e-3 * torch.randn(*shape, generator=gen)).to(torch.bfloat16)
    dev = torch.device("cuda", torch.cuda.device_count() - 1)
    p, b = p0.to(dev), b0.to(dev)
    muon.step_noalloc(p, g.to(dev), b, momentum=0.95, lr=0.02, weight_decay=0.01)
    torch.cuda.synchronize(dev)
    _check_against_oracle(p0, g, b0, p, b)
