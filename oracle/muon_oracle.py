"""CPU float64 oracle of the Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` use it.  It shares no code with the CUDA path.

It restates, in plain numpy float64 with no blocking, fusion or reordering,
what the pages describe.  The pages cited below are:

* [PG] "parameter-golf train_gpt.py 源码精读：Muon 优化器、Int8 量化与 DDP
  数据加载全解", part 1 "Muon 优化器是如何工作的":
  - section "核心思想：把矩阵梯度'正交化'" gives the Newton-Schulz function:
    cast to bf16, divide by the Frobenius norm, then ``steps`` rounds of
    A = X X^T; B = b A + c A A; X = a X + B X;
  - section "分布式细节：每个 rank 只算 1/N 的参数" gives the shape rescale
    factor max(1, m/n)^(1/2) on the NS result.
* [MCS] "Muon Custom Sizing 实战：modded-nanogpt 将注意力与 MLP 参数合并进同一
  reduce_scatter 调用，把 124M GPT 训练压进 150 秒":
  - section 2.3 gives ``(a, b, c) = (3.4445, -4.7750, 2.0315)``, five rounds;
  - section 四 (second pass) gives the momentum pair: the buffer moves towards
    the gradient by 1 - momentum, then the gradient moves towards the updated
    buffer by momentum (Nesterov); the decoupled decay by the factor
    1 - lr * wd on the parameter; and the NS result added with weight
    -lr * rescale.

Readings taken where the pages are silent or loose (each is listed in the
design notes with its reason):

* eps: the page's loop divides by the norm alone; here the divisor is
  ``||X||_F + eps`` so that a zero update gives X = 0 instead of NaN.
* norm kind: [MCS] speaks of the spectral norm, [PG]'s code takes the
  Frobenius norm.  The code wins: Frobenius.
* orientation: when rows > cols the iteration runs on the transpose and the
  result is transposed back (the Gram matrix is then the smaller m x m one).
* rescale: ``max(1, rows/cols) ** 0.5`` with rows/cols of the matrix handed
  to the step; a positive ``lr_scale`` argument overrides it.
* decay: multiplicative ``p * (1 - lr * wd)`` on the pre-update parameter.
* precision: everything here is float64 with no intermediate rounding; the
  pages' bf16 is the GPU path's business, and the parity tolerance absorbs it.

Parity pins (tests/test_oracle_pins.py): every function below is pinned to
something other than itself -- the SVD closed form of the iteration, exact
rational constants of the scalar polynomial, invariants, special cases and
brute force on tiny inputs.  No function here is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

# [MCS] section 2.3: the quintic coefficients, and five rounds
# ([PG] section 核心思想 also says the projection takes 5 steps).
NS5_COEFFS = (3.4445, -4.7750, 2.0315)
NS5_STEPS = 5
# Reading: divisor ||X||_F + eps (the printed loop has no eps).
NS5_EPS = 1e-7


def _f64(x) -> np.ndarray:
    return np.array(x, dtype=np.float64, copy=True)


def momentum_buffer_update(buf, grad, momentum: float) -> np.ndarray:
    """buf + (1 - momentum) * (grad - buf): the buffer moved towards the gradient.

    [MCS] section 四, second pass: the momentum buffer is lerped towards the
    gradient by weight ``1 - momentum`` before the Nesterov blend.
    """
    buf = _f64(buf)
    grad = _f64(grad)
    return buf + (1.0 - momentum) * (grad - buf)


def nesterov_blend(grad, buf, momentum: float) -> np.ndarray:
    """grad + momentum * (buf - grad): the Nesterov blend.

    [MCS] section 四: the gradient moved towards the momentum buffer by
    ``momentum``, taken with the buffer already updated.
    """
    grad = _f64(grad)
    buf = _f64(buf)
    return grad + momentum * (buf - grad)


def frobenius_normalise(X, eps: float = NS5_EPS) -> np.ndarray:
    """X / (||X||_F + eps).  [PG] section 核心思想: one Frobenius normalisation."""
    X = _f64(X)
    return X / (np.sqrt(np.sum(X * X)) + eps)


def newton_schulz5(G, steps: int = NS5_STEPS, coeffs=NS5_COEFFS,
                   eps: float = NS5_EPS) -> np.ndarray:
    """The quintic Newton-Schulz iteration on one 2-D matrix, in float64.

    [PG] section 核心思想: normalise once, then ``steps`` rounds of
    A = X X^T;  B = b A + c (A A);  X = a X + B X.
    The iteration runs on G^T when G has more rows than columns, and the
    result is transposed back, so that A is the smaller Gram matrix.
    """
    X = _f64(G)
    if X.ndim != 2:
        raise ValueError("newton_schulz5 takes one 2-D matrix")
    a, b, c = (float(v) for v in coeffs)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X = frobenius_normalise(X, eps)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    if transposed:
        X = X.T
    return X


def rescale_factor(rows: int, cols: int) -> float:
    """max(1, rows/cols) ** 0.5.  [PG] section 分布式细节: the shape rescale of the NS result."""
    return max(1.0, rows / cols) ** 0.5


def apply_update(param, O, lr: float, weight_decay: float,
                 lr_scale: float) -> np.ndarray:
    """p * (1 - lr * wd) - lr * lr_scale * O.

    [MCS] section 四: decay by lr * wd on the parameter, then the NS result
    added with weight -lr * rescale.
    """
    p = _f64(param)
    return (1.0 - lr * weight_decay) * p - (lr * lr_scale) * _f64(O)


def muon_step(param, grad, buf, *, momentum: float, nesterov: bool = True,
              lr: float, weight_decay: float, lr_scale: float = 0.0,
              steps: int = NS5_STEPS, coeffs=NS5_COEFFS,
              eps: float = NS5_EPS):
    """One Muon step on one 2-D weight.

    Returns (new_param, new_buf, O) with O the orthogonalised update before
    the learning-rate scaling.  ``lr_scale <= 0`` selects rescale_factor().
    """
    grad = _f64(grad)
    new_buf = momentum_buffer_update(buf, grad, momentum)
    u = nesterov_blend(grad, new_buf, momentum) if nesterov else new_buf
    O = newton_schulz5(u, steps, coeffs, eps)
    rows, cols = grad.shape
    scale = rescale_factor(rows, cols) if lr_scale <= 0 else float(lr_scale)
    new_param = apply_update(param, O, lr, weight_decay, scale)
    return new_param, new_buf, O


def muon_step_batched(params, grads, bufs, **kw):
    """muon_step over a stack [batch, rows, cols] of same-shape weights.

    [MCS] section 四 stacks the gradients of one parameter group into one
    batch; every matrix of the batch is independent.
    """
    params = _f64(params)
    grads = _f64(grads)
    bufs = _f64(bufs)
    out_p = np.empty_like(params)
    out_b = np.empty_like(bufs)
    out_o = np.empty_like(grads)
    for i in range(grads.shape[0]):
        out_p[i], out_b[i], out_o[i] = muon_step(params[i], grads[i], bufs[i], **kw)
    return out_p, out_b, out_o


def newton_schulz5_batched(G, steps: int = NS5_STEPS, coeffs=NS5_COEFFS,
                           eps: float = NS5_EPS) -> np.ndarray:
    """newton_schulz5 applied to each matrix of a [batch, rows, cols] stack."""
    G = _f64(G)
    return np.stack([newton_schulz5(G[i], steps, coeffs, eps)
                     for i in range(G.shape[0])]) if G.shape[0] else G.copy()
