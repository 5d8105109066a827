"""CPU float64 oracle of the Adam half of the optimizer -- test infrastructure only.

Nothing in the product path may import, call or execute this module (the same
rule as muon_oracle).  It restates, in numpy float64, the per-parameter update
of the DistAdam optimizer that trains the non-matrix parameters (embeddings,
head, scalars) next to Muon, as printed in

* [P3] "将 Adam 梯度同步（Reduce-Scatter）移入反向 Hook：modded-nanogpt 分布式优化器
  每步提速约 0.7 秒的工程实践", section 改动二 (step() 逆序遍历): per parameter
  slice, step counter t += 1; if wd != 0 the slice is multiplied by
  1 - lr * wd; exp_avg.mul_(beta1).add_(g, alpha = 1 - beta1);
  exp_avg_sq.mul_(beta2).addcmul_(g, g, value = 1 - beta2);
  bias1 = 1 - beta1 ** t; bias2 = 1 - beta2 ** t;
  denom = exp_avg_sq.sqrt() + eps; step_size = lr * sqrt(bias2) / bias1;
  p -= step_size * exp_avg / denom.
* [MCS] "Muon Custom Sizing 实战", section 四: the training script's DistAdam
  hyper-parameters lr = 0.008, betas = (0.8, 0.95), eps = 1e-8.

On one GPU the reduce-scatter / all-gather around the update (the subject of
[P3]) has nothing to do: each parameter is updated whole.  Readings: lr_scale
and wd_scale stand for the per-parameter ``lr_mul`` / ``wd_mul`` attributes
(1.0 when absent); the decay uses the scaled lr, as the printed code does.

Pins: tests/test_adam_oracle_pins.py (first-step closed form, brute-force scalar
recurrences, decay-only and zero-gradient cases, planted mistakes).
"""

from __future__ import annotations

import numpy as np

# [MCS] section 四: DistAdam settings of the training script.
ADAM_LR = 0.008
ADAM_BETAS = (0.8, 0.95)
ADAM_EPS = 1e-8


def _f64(x) -> np.ndarray:
    return np.array(x, dtype=np.float64, copy=True)


def adam_step(param, grad, exp_avg, exp_avg_sq, *, step: int, lr: float = ADAM_LR,
              betas=ADAM_BETAS, eps: float = ADAM_EPS, weight_decay: float = 0.0,
              lr_scale: float = 1.0, wd_scale: float = 1.0):
    """One DistAdam update of one parameter; `step` is t after its increment (t >= 1).

    Returns (new_param, new_exp_avg, new_exp_avg_sq).
    """
    if step < 1:
        raise ValueError("step counts from 1")
    p = _f64(param)
    g = _f64(grad)
    m = _f64(exp_avg)
    v = _f64(exp_avg_sq)
    beta1, beta2 = (float(b) for b in betas)
    lr_eff = lr * lr_scale
    if weight_decay != 0:
        p = p * (1.0 - lr_eff * weight_decay * wd_scale)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    bias1 = 1.0 - beta1 ** step
    bias2 = 1.0 - beta2 ** step
    denom = np.sqrt(v) + eps
    step_size = lr_eff * (np.sqrt(bias2) / bias1)
    p = p - step_size * (m / denom)
    return p, m, v
