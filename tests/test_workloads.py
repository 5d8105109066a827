"""Host checks of the seeded workload generator (shapes, seeds, determinism)."""

import torch

import workloads


def test_workload_shapes_match_descriptions():
    w = workloads.get("cfg3")
    shapes = [(g.batch, g.rows, g.cols) for g in w.groups]
    assert shapes == [(1, 1, 12), (10, 12, 768), (40, 768, 768), (11, 768, 3072), (11, 3072, 768)]
    assert w.n_matrices == 73
    assert workloads.get("cfg1").groups[0].rows == 128
    assert workloads.get("cfg2").momentum == 0.85
    assert workloads.get("cfg5").buf_std == 0.02
    assert workloads.get("cfg4").heavy_row_frac == 0.01


def test_draws_are_deterministic_and_distinct():
    w = workloads.get("cfg2")
    p1, g1, b1 = workloads.draw_stored_matrix(w, 1, 3)
    p2, g2, b2 = workloads.draw_stored_matrix(w, 1, 3)
    assert torch.equal(p1, p2) and torch.equal(g1, g2) and torch.equal(b1, b2)
    p3, g3, _ = workloads.draw_stored_matrix(w, 1, 4)
    assert not torch.equal(g1, g3) and not torch.equal(p1, p3)
    assert g1.dtype == torch.bfloat16 and p1.dtype == torch.float32
    assert torch.count_nonzero(b1) == 0


def test_qkvo_view_is_a_reinterpretation_of_the_stored_weight():
    w = workloads.get("cfg3")
    gi = [g.name for g in w.groups].index("attn_qkvo")
    P, G, B = workloads.make_group(w, gi)
    assert P.shape == (40, 768, 768) and P.is_contiguous()
    p0, g0, _ = workloads.draw_stored_matrix(w, gi, 0)
    assert p0.shape == (768, 3072)
    assert torch.equal(P[:4].reshape(768, 3072), p0)
    assert torch.equal(G[:4].reshape(768, 3072), g0)


def test_heavy_rows():
    w = workloads.Workload(name="t", description="", seed=9, groups=(workloads.Group("x", 2, 200, 64),),
                           grad_dtype=torch.float32, grad_std=1.0, momentum=0.9, heavy_row_frac=0.01)
    _, g, _ = workloads.draw_stored_matrix(w, 0, 0)
    row_norms = g.norm(dim=1)
    assert (row_norms > 20 * row_norms.median()).sum() == 2   # ceil(1% of 200)


def test_sample_indices():
    assert workloads.sample_indices(1) == [0]
    assert workloads.sample_indices(40) == [0, 20, 39]
    assert workloads.sample_indices(0) == []
