"""Seeded synthetic workloads for the Muon step: shapes, hyper-parameters, tensors.

This module holds none of the method's arithmetic.  It only says which
matrices a workload has and draws their seeded random contents; the CUDA
path's tests and benchmark and the CPU oracle's tests both take their inputs
from here (the oracle is then fed the exact bytes the GPU sees).

Recipe (one generator per matrix and per tensor kind):
  seed(matrix i, kind k) = workload.seed * 10_000_000 + 4 * i + k
  k = 0 gradient, 1 parameter, 2 momentum buffer, 3 heavy-row permutation
  i counts the stored matrices of the workload in group order.
Gradients are drawn in fp32 as N(0, grad_std), optionally with a fraction of
rows scaled (heavy-tailed singular values), then cast to the gradient dtype.
Parameters are fp32 N(0, param_std); momentum buffers are zeros or fp32
N(0, buf_std).  Values drawn on "cpu" and on "cuda" differ (different torch
generators); a test always draws on one device and copies bytes to the other.

Shapes follow the GPT models the pages train: the d=768 GPT-2 124M stack of
the modded-nanogpt record, whose attention weight is stored as (hdim, 4*dim)
and viewed as four (hdim, dim) blocks (Q, K, V, O) before orthogonalisation,
and the 9-layer d=512 model of parameter-golf.

The Adam half of the optimizer takes the parameters Muon does not: for the
GPT-2 124M stack the token embedding and the output head (vocab 50257 x 768
each, the sizes of that page's model) and a small vector of scalars (64
entries: the count is not printed).  Their seeds are
  seed(tensor i, kind k) = workload.seed * 10_000_000 + 5_000_000 + 4 * i + k
  k = 0 gradient, 1 parameter, 2 exp_avg, 3 exp_avg_sq.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Group:
    """`batch` same-shape matrices of `rows` x `cols`, stored contiguously.

    `stored` is the (count, rows, cols) shape the weights are kept in when it
    differs from the batch view (the QKVO attention weight).
    """
    name: str
    batch: int
    rows: int
    cols: int
    stored: tuple | None = None

    @property
    def stored_shape(self):
        return self.stored or (self.batch, self.rows, self.cols)


@dataclass(frozen=True)
class AdamTensor:
    """One parameter trained by the Adam half of the optimizer (flat, any shape)."""
    name: str
    shape: tuple
    lr_scale: float = 1.0
    wd_scale: float = 1.0

    @property
    def numel(self):
        return math.prod(self.shape)


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    seed: int
    groups: tuple
    grad_dtype: torch.dtype
    grad_std: float
    momentum: float
    lr: float = 0.02
    weight_decay: float = 0.01
    param_std: float = 0.02
    buf_std: float = 0.0
    heavy_row_frac: float = 0.0
    heavy_row_scale: float = 100.0
    steps: int = 5
    nesterov: bool = True
    adam: tuple = ()          # AdamTensor entries: embeddings, head, scalars
    adam_step: int = 100      # Adam step count t of the drawn state

    @property
    def adam_numel(self):
        return sum(t.numel for t in self.adam)

    @property
    def n_matrices(self):
        return sum(g.batch for g in self.groups)

    @property
    def n_elements(self):
        return sum(g.batch * g.rows * g.cols for g in self.groups)


_W = [
    Workload(
        name="single-128x256",
        description="one fp32 gradient 128x256 ~N(0,1), zero momentum buffer",
        seed=0, groups=(Group("G", 1, 128, 256),),
        grad_dtype=torch.float32, grad_std=1.0, momentum=0.95),
    Workload(
        name="gpt-9L-d512",
        description="9-layer d=512 GPT (8 heads, 4 KV heads): c_q+proj 512x512, c_k+c_v 256x512, "
                    "fc 1024x512, mlp proj 512x1024; bf16 grads ~N(0,1e-3), momentum 0.85",
        seed=2,
        groups=(Group("c_q+proj", 18, 512, 512), Group("c_k+c_v", 18, 256, 512),
                Group("fc", 9, 1024, 512), Group("mlp_proj", 9, 512, 1024)),
        grad_dtype=torch.bfloat16, grad_std=1e-3, momentum=0.85),
    Workload(
        name="gpt2-124M-d768",
        description="GPT-2 124M d=768: 10 QKVO weights (768x3072 viewed as 4x768x768), "
                    "11x 768x3072 + 11x 3072x768 MLP, 10 attn_gate 12x768, 1 smear_gate 1x12; "
                    "bf16 grads ~N(0,1e-3), momentum 0.95",
        seed=3,
        groups=(Group("smear_gate", 1, 1, 12), Group("attn_gate", 10, 12, 768),
                Group("attn_qkvo", 40, 768, 768, stored=(10, 768, 3072)),
                Group("mlp_fc", 11, 768, 3072), Group("mlp_proj", 11, 3072, 768)),
        grad_dtype=torch.bfloat16, grad_std=1e-3, momentum=0.95,
        adam=(AdamTensor("embed", (50257, 768)), AdamTensor("lm_head", (50257, 768)),
              AdamTensor("scalars", (64,)))),
    Workload(
        name="gpt-24L-d2048",
        description="24-layer d=2048 GPT: 96 attn 2048x2048, 24 MLP-up 8192x2048, 24 MLP-down "
                    "2048x8192; bf16 grads ~N(0,1e-3) with 1% of rows x100",
        seed=4,
        groups=(Group("attn", 96, 2048, 2048), Group("mlp_up", 24, 8192, 2048),
                Group("mlp_down", 24, 2048, 8192)),
        grad_dtype=torch.bfloat16, grad_std=1e-3, momentum=0.95, heavy_row_frac=0.01),
    Workload(
        name="gpt-32L-d4096",
        description="32-layer d=4096 GPT: 128 attn 4096x4096, 32 each of 11008x4096 (up), "
                    "4096x11008 (down), 11008x4096 (gate); bf16 grads ~N(0,1e-3), "
                    "fp32 momentum ~N(0,0.02)",
        seed=5,
        groups=(Group("attn", 128, 4096, 4096), Group("mlp_up", 32, 11008, 4096),
                Group("mlp_down", 32, 4096, 11008), Group("mlp_gate", 32, 11008, 4096)),
        grad_dtype=torch.bfloat16, grad_std=1e-3, momentum=0.95, buf_std=0.02),
]

WORKLOADS = {w.name: w for w in _W}
# short aliases in the order the workloads are listed
ALIASES = {f"cfg{i + 1}": w.name for i, w in enumerate(_W)}


def get(name: str) -> Workload:
    return WORKLOADS[ALIASES.get(name, name)]


def matrix_seed(wl: Workload, matrix_index: int, kind: int) -> int:
    return wl.seed * 10_000_000 + 4 * matrix_index + kind


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _stored_offsets(wl: Workload):
    """First stored-matrix index of each group."""
    out, i = [], 0
    for g in wl.groups:
        out.append(i)
        i += g.stored_shape[0]
    return out


def draw_stored_matrix(wl: Workload, group_index: int, j: int, device="cpu"):
    """(param fp32, grad, buf fp32) of stored matrix j of a group, each (rows, cols) as stored."""
    grp = wl.groups[group_index]
    _, r, c = grp.stored_shape
    i = _stored_offsets(wl)[group_index] + j
    g = torch.randn(r, c, generator=_gen(device, matrix_seed(wl, i, 0)), device=device,
                    dtype=torch.float32) * wl.grad_std
    if wl.heavy_row_frac > 0:
        k = math.ceil(wl.heavy_row_frac * r)
        rows = torch.randperm(r, generator=_gen(device, matrix_seed(wl, i, 3)), device=device)[:k]
        g[rows] *= wl.heavy_row_scale
    g = g.to(wl.grad_dtype)
    p = torch.randn(r, c, generator=_gen(device, matrix_seed(wl, i, 1)), device=device,
                    dtype=torch.float32) * wl.param_std
    if wl.buf_std > 0:
        b = torch.randn(r, c, generator=_gen(device, matrix_seed(wl, i, 2)), device=device,
                        dtype=torch.float32) * wl.buf_std
    else:
        b = torch.zeros(r, c, device=device, dtype=torch.float32)
    return p, g, b


def make_group(wl: Workload, group_index: int, device="cpu"):
    """Contiguous (params, grads, bufs), each viewed as [batch, rows, cols]."""
    grp = wl.groups[group_index]
    n, r, c = grp.stored_shape
    P = torch.empty(n, r, c, device=device, dtype=torch.float32)
    G = torch.empty(n, r, c, device=device, dtype=wl.grad_dtype)
    B = torch.empty(n, r, c, device=device, dtype=torch.float32)
    for j in range(n):
        p, g, b = draw_stored_matrix(wl, group_index, j, device)
        P[j].copy_(p)
        G[j].copy_(g)
        B[j].copy_(b)
    shape = (grp.batch, grp.rows, grp.cols)
    return P.view(shape), G.view(shape), B.view(shape)


def make_workload(wl: Workload, device="cpu"):
    """List of (Group, params, grads, bufs) for every group of the workload."""
    return [(grp, *make_group(wl, gi, device)) for gi, grp in enumerate(wl.groups)]


def adam_seed(wl: Workload, tensor_index: int, kind: int) -> int:
    return wl.seed * 10_000_000 + 5_000_000 + 4 * tensor_index + kind


def draw_adam_tensor(wl: Workload, index: int, device="cpu", spec: AdamTensor | None = None):
    """(param fp32, grad, exp_avg fp32, exp_avg_sq fp32) of one Adam tensor, flat.

    Mid-training state: grad ~ N(0, grad_std) in the workload's gradient dtype,
    param ~ N(0, param_std), exp_avg ~ N(0, grad_std), exp_avg_sq = N(0, grad_std)^2.
    """
    spec = spec or wl.adam[index]
    n = spec.numel
    g = (torch.randn(n, generator=_gen(device, adam_seed(wl, index, 0)), device=device)
         * wl.grad_std).to(wl.grad_dtype)
    p = torch.randn(n, generator=_gen(device, adam_seed(wl, index, 1)), device=device) * wl.param_std
    m = torch.randn(n, generator=_gen(device, adam_seed(wl, index, 2)), device=device) * wl.grad_std
    v = (torch.randn(n, generator=_gen(device, adam_seed(wl, index, 3)), device=device)
         * wl.grad_std) ** 2
    return p, g, m, v


def make_adam_set(wl: Workload, device="cpu"):
    """List of (AdamTensor, param, grad, exp_avg, exp_avg_sq) of the workload."""
    return [(t, *draw_adam_tensor(wl, i, device)) for i, t in enumerate(wl.adam)]


def sample_indices(batch: int):
    """Deterministic subset of a batch checked against the oracle: first, middle, last."""
    return sorted({0, batch // 2, batch - 1}) if batch > 0 else []
