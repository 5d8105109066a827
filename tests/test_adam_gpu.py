"""GPU parity of the DistAdam update kernel against the float64 oracle.

Inputs are drawn on the CPU, copied to the GPU, updated there through the C ABI
(muon_adam_step), and compared element by element with the oracle fed the same
bytes.  Bar: relative Frobenius error <= 1e-5 on param, exp_avg and exp_avg_sq
(the fp32 elementwise tolerance), and on the parameter change itself
||dp_gpu - dp_ref|| <= 1e-5 ||dp_ref|| + 2^-23 ||p|| (the second term is the
rounding of the fp32 parameter the change is added to).
"""

import math

import numpy as np
import pytest
import torch

import newton_schulz_step_gb300 as muon
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _rel(a, b):
    b = np.asarray(b, dtype=np.float64)
    d = np.linalg.norm(np.asarray(a, dtype=np.float64) - b)
    n = np.linalg.norm(b)
    return d / n if n > 0 else d


def _draw(n, seed, g_dtype, scale=1e-3):
    gen = torch.Generator().manual_seed(seed)
    p = torch.randn(n, generator=gen) * 0.02
    g = (torch.randn(n, generator=gen) * scale).to(g_dtype)
    m = torch.randn(n, generator=gen) * scale
    v = (torch.randn(n, generator=gen) * scale) ** 2
    return p, g, m, v


def _check(cpu, gpu, step, *, lr, betas, eps, wd, scales):
    for (p, g, m, v), (pd, gd, md, vd), (ls, ws) in zip(cpu, gpu, scales):
        rp, rm, rv = oracle.adam_step(p.double().numpy(), g.double().numpy(), m.double().numpy(),
                                      v.double().numpy(), step=step, lr=lr, betas=betas, eps=eps,
                                      weight_decay=wd, lr_scale=ls, wd_scale=ws)
        gp, gm, gv = (x.cpu().double().numpy() for x in (pd, md, vd))
        assert _rel(gm, rm) <= TOL, ("exp_avg", p.numel(), _rel(gm, rm))
        assert _rel(gv, rv) <= TOL, ("exp_avg_sq", p.numel(), _rel(gv, rv))
        assert _rel(gp, rp) <= TOL, ("param", p.numel(), _rel(gp, rp))
        p0 = p.double().numpy()
        dref, dgpu = rp - p0, gp - p0
        bound = TOL * np.linalg.norm(dref) + 2.0 ** -23 * np.linalg.norm(p0)
        assert np.linalg.norm(dgpu - dref) <= bound, ("dp", p.numel())


# ragged sizes around the 4096-element unit and the 4-element vector
SIZES = [1, 3, 4, 5, 4095, 4096, 4097, 8191, 12345, 3 * 4096 + 6]


@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("step,wd", [(1, 0.0), (2, 0.1), (10, 0.0), (1000, 0.05)])
def test_ragged_tensors_match_oracle(g_dtype, step, wd):
    lr, betas, eps = oracle.ADAM_LR, oracle.ADAM_BETAS, oracle.ADAM_EPS
    cpu = [_draw(n, 100 + i, g_dtype) for i, n in enumerate(SIZES)]
    gpu = [tuple(x.cuda() for x in t) for t in cpu]
    scales = [(1.0 + 0.25 * (i % 3), 1.0 - 0.3 * (i % 2)) for i in range(len(SIZES))]
    muon.adam_step([(*t, ls, ws) for t, (ls, ws) in zip(gpu, scales)], step, lr=lr, betas=betas,
                   eps=eps, weight_decay=wd)
    torch.cuda.synchronize()
    _check(cpu, gpu, step, lr=lr, betas=betas, eps=eps, wd=wd, scales=scales)


def test_more_tensors_than_one_launch_takes():
    # 70 tensors: two launches of up to 64 each
    cpu = [_draw(17 + 61 * i, 900 + i, torch.bfloat16) for i in range(70)]
    gpu = [tuple(x.cuda() for x in t) for t in cpu]
    before = muon.kernel_launch_count()
    muon.adam_step(gpu, 3, weight_decay=0.01)
    torch.cuda.synchronize()
    assert muon.kernel_launch_count() - before == 2
    _check(cpu, gpu, 3, lr=oracle.ADAM_LR, betas=oracle.ADAM_BETAS, eps=oracle.ADAM_EPS, wd=0.01,
           scales=[(1.0, 1.0)] * 70)


def test_zero_state_first_step_is_sign_like():
    # t = 1 from zero moments: p1 = p0 - lr g / (|g| + eps / sqrt(1 - b2)), each |step| < lr
    n = 10000
    p, g, _, _ = _draw(n, 7, torch.float32)
    z = torch.zeros(n)
    gpu = [(p.cuda(), g.cuda(), z.cuda(), z.cuda())]
    muon.adam_step(gpu, 1)
    torch.cuda.synchronize()
    _check([(p, g, z, z)], gpu, 1, lr=oracle.ADAM_LR, betas=oracle.ADAM_BETAS,
           eps=oracle.ADAM_EPS, wd=0.0, scales=[(1.0, 1.0)])
    step = (gpu[0][0].cpu() - p).abs()
    assert float(step.max()) <= oracle.ADAM_LR * (1 + 1e-6)


def test_zero_gradient_and_zero_state_is_pure_decay():
    n = 4096 + 3
    p = torch.randn(n)
    z = torch.zeros(n)
    gpu = [(p.cuda(), z.cuda(), z.cuda(), z.cuda(), 2.0, 0.5)]
    muon.adam_step(gpu, 5, lr=0.01, weight_decay=0.3)
    torch.cuda.synchronize()
    expect = p.double() * (1 - 0.01 * 2.0 * 0.3 * 0.5)
    assert _rel(gpu[0][0].cpu().double().numpy(), expect.numpy()) <= 2e-7
    assert torch.count_nonzero(gpu[0][2]) == 0 and torch.count_nonzero(gpu[0][3]) == 0


def test_state_carries_over_several_steps():
    # three consecutive steps with fresh gradients: the kernel's state feeds the next step
    n = 3 * 4096 + 11
    p, _, m, v = _draw(n, 11, torch.float32)
    P, M, V = p.double().numpy(), m.double().numpy(), v.double().numpy()
    dev = [p.cuda(), None, m.cuda(), v.cuda()]
    for t in (1, 2, 3):
        g = (torch.randn(n, generator=torch.Generator().manual_seed(50 + t)) * 1e-3).to(
            torch.bfloat16)
        dev[1] = g.cuda()
        muon.adam_step([tuple(dev)], t, weight_decay=0.02)
        P, M, V = oracle.adam_step(P, g.double().numpy(), M, V, step=t, weight_decay=0.02)
    torch.cuda.synchronize()
    assert _rel(dev[0].cpu().double().numpy(), P) <= TOL
    assert _rel(dev[2].cpu().double().numpy(), M) <= TOL
    assert _rel(dev[3].cpu().double().numpy(), V) <= TOL


def test_empty_and_skipped_tensors():
    before = muon.kernel_launch_count()
    muon.adam_step([], 1)
    e = torch.empty(0, device="cuda")
    muon.adam_step([(e, e, e, e)], 1)
    assert muon.kernel_launch_count() == before


def test_gpt2_124m_adam_set_full_size():
    # the embedding and head of the GPT-2 124M model (50257 x 768 each) plus scalars,
    # in the launch configuration the benchmark times; the whole arrays are compared
    wl = workloads.get("gpt2-124M-d768")
    sets = workloads.make_adam_set(wl)
    cpu = [(p, g, m, v) for _, p, g, m, v in sets]
    gpu = [tuple(x.cuda() for x in t) for t in cpu]
    scales = [(t.lr_scale, t.wd_scale) for t, *_ in sets]
    muon.AdamStep([(*t, ls, ws) for t, (ls, ws) in zip(gpu, scales)],
                  weight_decay=0.0)(wl.adam_step)
    torch.cuda.synchronize()
    _check(cpu, gpu, wl.adam_step, lr=oracle.ADAM_LR, betas=oracle.ADAM_BETAS,
           eps=oracle.ADAM_EPS, wd=0.0, scales=scales)
    assert math.isfinite(float(gpu[0][0].sum()))
