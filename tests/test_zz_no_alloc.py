"""lei_inject_noalloc against lei_inject, through the C ABI.

lei_inject_noalloc serves callers that cannot allocate device memory where
LEI is applied (a framework whose caching allocator owns the pool, a fixed
device-memory budget, no allocator at the call site): it keeps its scratch in
a fixed array inside the library instead of taking a workspace.  Its results
must equal lei_inject's within the LEI tolerance, call after call (the shared
scratch keeps the previous call's contents).  This file is collected last so
that a failure here stops a -x run only after every other test has run; it
also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LEI_ABS_TOL = 1e-6


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _case(N, E, k, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    r = torch.rand(N, E, generator=g, device="cuda")
    topk = torch.topk(r, k, dim=1).indices.to(torch.int32)
    topk[: N // 4] = torch.arange(k, dtype=torch.int32, device="cuda")  # imbalance
    grad = torch.randn(N, E, generator=g, device="cuda") * 1e-3
    return grad, topk.contiguous()


def test_noalloc_matches_workspace_version_twice_in_a_row(qb):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(65536, 256, 6, 32768, 8e-5, 1), (4097, 64, 8, 1000, 0.5, 2)]
    for N, E, k, bt, eta, seed in cases:
        grad, topk = _case(N, E, k, seed)
        g_ref = grad.clone()
        g_new = grad.clone()
        nb = (N + bt - 1) // bt
        ws = torch.empty(nb, E, dtype=torch.float32, device="cuda")
        st = qb.lib.lei_inject(ctypes.c_void_p(g_ref.data_ptr()), ctypes.c_void_p(topk.data_ptr()),
                               N, E, k, eta, bt, ctypes.c_void_p(ws.data_ptr()), stream)
        assert st == qb.QB_OK
        st = qb.lib.lei_inject_noalloc(ctypes.c_void_p(g_new.data_ptr()),
                                       ctypes.c_void_p(topk.data_ptr()), N, E, k, eta, bt, stream)
        assert st == qb.QB_OK
        torch.cuda.synchronize()
        diff = (g_new - g_ref).abs().max().item()
        assert diff <= LEI_ABS_TOL
        assert not torch.equal(g_new, grad)  # the call did change the gradient


def test_noalloc_rejects_sizes_beyond_its_scratch(qb):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    grad, topk = _case(300, 256, 6, 3)
    before = grad.clone()
    # 300 batches of one token x 256 experts = 76800 floats > 65536
    st = qb.lib.lei_inject_noalloc(ctypes.c_void_p(grad.data_ptr()),
                                   ctypes.c_void_p(topk.data_ptr()), 300, 256, 6, 8e-5, 1, stream)
    assert st == qb.QB_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(grad, before)
    # 256 batches fit exactly
    st = qb.lib.lei_inject_noalloc(ctypes.c_void_p(grad.data_ptr()),
                                   ctypes.c_void_p(topk.data_ptr()), 256, 256, 6, 8e-5, 1, stream)
    assert st == qb.QB_OK
    torch.cuda.synchronize()
    assert np.isfinite(grad.cpu().numpy()).all()
