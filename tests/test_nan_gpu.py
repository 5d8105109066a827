"""Non-finite gradients on every path, against the oracle's pattern.

The pages put no guard in the step: a NaN or an Inf in a gradient spreads
through the Frobenius norm to the whole Newton-Schulz result of that matrix,
so the matrix's parameters all become NaN, while its momentum buffer is
non-finite only where the gradient was.  The other matrices of the same call
are untouched by it.  The GPU path must give the same pattern (TMA's zero
padding, the fp32 small-matrix kernel or the fused kernel's on-chip rounds must
not mask it), and the finite matrices must still match the oracle.
"""

import numpy as np
import pytest
import torch

import newton_schulz_step_gb300 as muon
import oracle

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2
SMALL_TOL = 1e-4
EW_TOL = 1e-5

# shape (batch 3: matrix 0 finite, matrix 1 one NaN, matrix 2 one +Inf), rounds mode
CASES = [((3, 160, 288), 2, True), ((3, 300, 520), 1, True), ((3, 300, 520), 0, True),
         ((3, 520, 300), 1, True), ((3, 256, 640), 1, True), ((3, 256, 640), 0, True),
         ((3, 12, 96), 2, True), ((3, 160, 288), 2, False)]
IDS = ["fused", "persistent", "per-stage", "persistent-tall", "streamed-persistent",
       "streamed-per-stage", "small", "staged-in-fused-range"]


def rel(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.mark.parametrize("shape,rounds,fused", CASES, ids=IDS)
def test_nan_and_inf_gradients_follow_the_oracle_pattern(shape, rounds, fused):
    gen = torch.Generator().manual_seed(5)
    p0 = 0.02 * torch.randn(*shape, generator=gen)
    g0 = (1e-3 * torch.randn(*shape, generator=gen)).to(torch.bfloat16)
    b0 = 0.02 * torch.randn(*shape, generator=gen)
    r, c = shape[1:]
    g0[1, r // 3, c // 2] = float("nan")
    g0[2, r - 1, 0] = float("inf")
    p, g, b = p0.cuda(), g0.cuda(), b0.cuda()
    with muon.persistent_rounds(rounds), muon.fused_ns(fused):
        muon.step(p, g, b, momentum=0.95, lr=0.02, weight_decay=0.01)
    torch.cuda.synchronize()
    p1, b1 = f64(p), f64(b)
    tol = SMALL_TOL if min(r, c) < 64 else NS_TOL
    with np.errstate(invalid="ignore", over="ignore"):
        for i in range(shape[0]):
            p_ref, b_ref, _ = oracle.muon_step(f64(p0[i]), f64(g0[i]), f64(b0[i]),
                                               momentum=0.95, lr=0.02, weight_decay=0.01)
            # the momentum buffer: non-finite exactly where the oracle's is, same values
            assert np.array_equal(np.isnan(b1[i]), np.isnan(b_ref)), i
            assert np.array_equal(np.isposinf(b1[i]), np.isposinf(b_ref)), i
            fin = np.isfinite(b_ref)
            assert rel(b1[i][fin], b_ref[fin]) < EW_TOL
            # the parameters: all NaN for a matrix with a non-finite gradient
            assert np.array_equal(np.isnan(p1[i]), np.isnan(p_ref)), i
            if i == 0:
                assert np.isfinite(p1[i]).all()
                upd, upd_ref = p1[i] - 0.9998 * f64(p0[i]), p_ref - 0.9998 * f64(p0[i])
                assert rel(upd, upd_ref) < tol
            else:
                assert np.isnan(p_ref).all() and np.isnan(p1[i]).all()
