"""The device status word and the bounded waits, through the C ABI.

Every wait of the kernels on an mbarrier is bounded: on giving up it sets
bit 0 of a device status word and the kernel returns instead of trapping or
spinning.  qb_selftest_wait_timeout runs that path on an mbarrier nothing
completes (with a short poll limit), so the reporting is tested without any
GPU fault: the flag is reported once by qb_device_status, which clears it,
and later calls run normally.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _status(qb):
    flags = ctypes.c_int(-1)
    st = qb.lib.qb_device_status(ctypes.byref(flags))
    return st, flags.value


def test_bounded_wait_gives_up_and_reports(qb, orc):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _status(qb) == (qb.QB_OK, 0)
    assert qb.lib.qb_selftest_wait_timeout(0, stream) == qb.QB_EINVAL
    assert qb.lib.qb_selftest_wait_timeout((1 << 24) + 1, stream) == qb.QB_EINVAL
    assert qb.lib.qb_selftest_wait_timeout(2000, stream) == qb.QB_OK
    torch.cuda.synchronize()
    assert _status(qb) == (qb.QB_EDEVICE, 1)  # the wait ran out and said so
    assert _status(qb) == (qb.QB_OK, 0)       # reading cleared it
    # the context is intact: a routing call afterwards is exact and clean
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], n_micro=1, n_tokens=1000)
    bias, mbs = inputs.router_layer(w, 11, device="cuda")
    hist = torch.zeros(w.E, 256, dtype=torch.int32, device="cuda")
    qb.qb_route_hist_hi(mbs[0], bias, w.k, hist)
    torch.cuda.synchronize()
    assert _status(qb) == (qb.QB_OK, 0)
    m = orc.route(mbs[0].cpu().numpy(), bias.cpu().numpy(), w.k, want=("margins",))["margins"]
    assert np.array_equal(hist.cpu().numpy(), orc.hist_hi(orc.keys(m)))
