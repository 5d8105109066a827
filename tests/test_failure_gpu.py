"""Failure handling on the GPU, without any fault or hang.

A bounded device-side wait that gives up records it in the workspace's sticky
status word.  The self-test entry point makes such a wait run out on purpose
(a barrier nothing completes, a 1 ms limit); these tests then check that every
kernel of a later call on that workspace returns at entry -- the call takes
milliseconds, not a 2 s wait per launch, and changes nothing -- and that the
workspace works normally once the word is cleared.
"""

import time

import numpy as np
import pytest
import torch

import newton_schulz_step_gb300 as muon
import oracle

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2
SMALL_TOL = 1e-4
NS5_SMALL_TOL = 5e-3
EW_TOL = 1e-5
TIMEOUT = 4  # MUON_ERR_TIMEOUT


def rel(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def f64(t):
    return t.detach().float().cpu().double().numpy()


def _rand(shape, std, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(dtype)


# (shape, persistent rounds mode): the staged path with one launch per stage and
# round (ns5: prologue + 15 GEMM launches + apply), the persistent rounds kernel,
# the fused kernel, and the fp32 small-matrix kernel
CASES = [((1, 300, 520), 0), ((1, 300, 520), 1), ((2, 160, 288), 2), ((3, 12, 96), 2)]
IDS = ["per-stage", "persistent", "fused", "small"]


@pytest.mark.parametrize("shape,rounds", CASES, ids=IDS)
def test_ns5_on_a_poisoned_workspace_returns_at_once_and_writes_nothing(shape, rounds):
    G = _rand(shape, 1.0, torch.bfloat16, 11).cuda()
    ws = muon.Workspace(muon.workspace_bytes(*shape))
    with muon.persistent_rounds(rounds):
        muon.ns5(G, workspace=ws)                 # warm: module load, tensor-map setup
        torch.cuda.synchronize()
        assert muon.workspace_status(ws) == 0
        muon.selftest_wait_timeout(ws, limit_us=1000)
        assert muon.workspace_status(ws) == TIMEOUT
        out = torch.full(shape, 7.0, dtype=torch.bfloat16, device="cuda")
        t0 = time.perf_counter()
        muon.ns5(G, out=out, workspace=ws)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert dt < 0.5, f"a call on a poisoned workspace took {dt:.3f} s"
        assert bool((out == 7.0).all()), "a call on a poisoned workspace wrote its output"
        assert muon.workspace_status(ws, clear=True) == TIMEOUT
        assert muon.workspace_status(ws) == 0
        muon.ns5(G, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert muon.workspace_status(ws) == 0
    # (the fp32 small-matrix result is returned in bf16: one rounding, ~2e-3)
    tol = NS5_SMALL_TOL if min(shape[1:]) < 64 else NS_TOL
    for i in range(shape[0]):
        assert rel(f64(out[i]), oracle.newton_schulz5(f64(G[i]))) < tol


# grouped steps: staged per-stage and persistent (parameter write after the NS),
# and the write streamed beside the persistent rounds kernel (cols % 8 == 0)
STEP_CASES = [([(1, 300, 520), (2, 12, 96)], 0), ([(1, 300, 520), (2, 12, 96)], 1),
              ([(2, 256, 640), (1, 640, 256)], 1), ([(2, 160, 288)], 2)]
STEP_IDS = ["per-stage", "persistent", "streamed", "fused"]


@pytest.mark.parametrize("shapes,rounds", STEP_CASES, ids=STEP_IDS)
def test_step_on_a_poisoned_workspace_changes_nothing(shapes, rounds):
    host = [(_rand(s, 0.02, torch.float32, 20 + 3 * k),
             _rand(s, 1e-3, torch.bfloat16, 21 + 3 * k),
             _rand(s, 0.02, torch.float32, 22 + 3 * k)) for k, s in enumerate(shapes)]
    dev = [(p.cuda(), g.cuda(), b.cuda()) for p, g, b in host]
    with muon.persistent_rounds(rounds):
        step = muon.GroupedStep(dev, momentum=0.95, lr=0.02, weight_decay=0.01)
        muon.selftest_wait_timeout(step.workspace, limit_us=1000)
        assert muon.workspace_status(step.workspace) == TIMEOUT
        t0 = time.perf_counter()
        step()
        step()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert dt < 0.5, f"two steps on a poisoned workspace took {dt:.3f} s"
        for (p0, _, b0), (p, _, b) in zip(host, dev):
            assert torch.equal(p.cpu(), p0) and torch.equal(b.cpu(), b0)
        assert muon.workspace_status(step.workspace, clear=True) == TIMEOUT
        step()
        torch.cuda.synchronize()
        assert muon.workspace_status(step.workspace) == 0
    for (p0, g0, b0), (p, _, b) in zip(host, dev):
        for i in range(p0.shape[0]):
            p_ref, b_ref, _ = oracle.muon_step(f64(p0[i]), f64(g0[i]), f64(b0[i]),
                                               momentum=0.95, lr=0.02, weight_decay=0.01)
            assert rel(f64(b[i]), b_ref) < EW_TOL
            tol = SMALL_TOL if min(p0.shape[1:]) < 64 else NS_TOL
            upd, upd_ref = f64(p[i]) - 0.9998 * f64(p0[i]), p_ref - 0.9998 * f64(p0[i])
            assert rel(upd, upd_ref) < tol
