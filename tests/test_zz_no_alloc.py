"""lei_inject_noalloc against lei_inject, through the C ABI.

lei_inject_noalloc serves callers that cannot allocate device memory where
LEI is applied (a framework whose caching allocator owns the pool, a fixed
device-memory budget, no allocator at the call site): it keeps its scratch in
a fixed array inside the library instead of taking a workspace.  It runs the
same kernels as lei_inject, so its results must equal lei_inject's bit for
bit, call after call (the shared scratch keeps the previous call's contents).
This file is collected last so that a failure here stops a -x run only after
every other test has run; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _case(N, E, k, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    r = torch.rand(N, E, generator=g, device="cuda")
    topk = torch.topk(r, k, dim=1).indices.to(torch.int32)
    topk[: N // 4] = torch.arange(k, dtype=torch.int32, device="cuda")  # imbalance
    grad = torch.randn(N, E, generator=g, device="cuda") * 1e-3
    return grad, topk.contiguous()


def _with_workspace(qb, grad, topk, eta, bt):
    N, E = grad.shape
    k = topk.shape[1]
    nb = (N + bt - 1) // bt
    ws = torch.empty(nb, E, dtype=torch.float32, device="cuda")
    out = grad.clone()
    st = qb.lib.lei_inject(_p(out), _p(topk), N, E, k, eta, bt, _p(ws), _stream())
    assert st == qb.QB_OK
    return out


def _noalloc(qb, grad, topk, eta, bt):
    N, E = grad.shape
    k = topk.shape[1]
    out = grad.clone()
    st = qb.lib.lei_inject_noalloc(_p(out), _p(topk), N, E, k, eta, bt, _stream())
    assert st == qb.QB_OK
    return out


def _bits(t):
    return t.contiguous().view(torch.int32)


def test_noalloc_bit_equal_to_workspace_version_on_repeated_calls(qb):
    # the second shape runs twice in a row after a call with another shape:
    # the shared scratch then holds the previous calls' values
    cases = [(65536, 256, 6, 32768, 8e-5, 1), (4097, 64, 8, 1000, 0.5, 2),
             (4097, 64, 8, 1000, 0.5, 2)]
    for N, E, k, bt, eta, seed in cases:
        grad, topk = _case(N, E, k, seed)
        ref = _with_workspace(qb, grad, topk, eta, bt)
        new = _noalloc(qb, grad, topk, eta, bt)
        torch.cuda.synchronize()
        assert torch.equal(_bits(new), _bits(ref))
        assert not torch.equal(new, grad)  # the call did change the gradient
    assert qb.device_status() == 0


def test_noalloc_at_capacity_and_beyond(qb, orc):
    grad, topk = _case(300, 256, 6, 3)
    before = grad.clone()
    # 300 batches of one token x 256 experts = 76800 floats > 65536: rejected
    st = qb.lib.lei_inject_noalloc(_p(grad), _p(topk), 300, 256, 6, 8e-5, 1, _stream())
    assert st == qb.QB_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(grad, before)
    # 256 batches of one token fill the scratch exactly
    g256, t256 = grad[:256].clone(), topk[:256].contiguous()
    ref = _with_workspace(qb, g256, t256, 8e-5, 1)
    new = _noalloc(qb, g256, t256, 8e-5, 1)
    torch.cuda.synchronize()
    assert torch.equal(_bits(new), _bits(ref))
    # and each one-token batch matches the oracle's LEI within its tolerance
    g_host, t_host = g256.cpu().numpy(), t256.cpu().numpy()
    want = np.empty_like(g_host)
    for i in range(256):
        want[i:i + 1] = orc.lei(g_host[i:i + 1], t_host[i:i + 1], 8e-5)[0]
    assert np.max(np.abs(new.cpu().numpy() - want)) <= 1e-6
    assert qb.device_status() == 0
