"""muon_step_noalloc (through the C ABI) against muon_step.

muon_step_noalloc serves callers that cannot allocate device memory (an
allocator that owns the whole GPU, a plug-in limited to the memory it is given,
a loop that forbids allocation after start-up): its scratch is an array built
into the library instead of a caller workspace.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import newton_schulz_step_gb300 as muon

pytestmark = pytest.mark.gpu

NS_TOL = 3e-2   # bf16 tensor-core NS, as in the parity tests
EW_TOL = 1e-5   # fp32 elementwise momentum buffer
SCRATCH = 64 << 20


def _rel(x, ref):
    x, ref = x.double().cpu().numpy(), ref.double().cpu().numpy()
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


@pytest.mark.parametrize("shape,gdt", [((4, 768, 3072), torch.bfloat16),
                                       ((3, 520, 300), torch.float32),
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
    a, b, c = muon.COEFFS
    stream = torch.cuda.current_stream().cuda_stream
    gdt_code = 1 if gdt == torch.bfloat16 else 0
    decay = 1 - 0.02 * 0.01
    for g in grads:                       # two calls in a row, state carried over
        p_before = p_ref.clone()
        code = L.muon_step(p_ref.data_ptr(), g.data_ptr(), gdt_code, b_ref.data_ptr(), *shape,
                           0.95, 1, 0.02, 0.01, 0.0, 5, a, b, c, 1e-7, ws.ptr, ws.nbytes, stream)
        assert code == 0, muon.status_string(code)
        code = L.muon_step_noalloc(p_new.data_ptr(), g.data_ptr(), gdt_code, b_new.data_ptr(),
                                   *shape, 0.95, 1, 0.02, 0.01, 0.0, 5, a, b, c, 1e-7, stream)
        assert code == 0, muon.status_string(code)
        torch.cuda.synchronize()
        assert _rel(b_new, b_ref) < EW_TOL
        assert _rel(p_new - decay * p_before, p_ref - decay * p_before) < NS_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = muon.load_library()
    shape = (1, 4096, 4096)                # needs ~134 MB of scratch
    assert L.muon_workspace_bytes(*shape) > SCRATCH
    a, b, c = muon.COEFFS
    # rejected before anything is enqueued: the pointers are never touched
    code = L.muon_step_noalloc(0x1000, 0x2000, 1, 0x3000, *shape, 0.95, 1, 0.02, 0.01, 0.0, 5,
                               a, b, c, 1e-7, None)
    assert code == 5   # MUON_ERR_WORKSPACE
