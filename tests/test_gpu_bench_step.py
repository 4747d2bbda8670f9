"""The benchmark's step schedule computes what the serial layer sequence does.

bench.py runs each layer's LEI rho kernel on a second stream beside the EQB
tail, and enqueues its grad update behind the next layer's hi pass as a
programmatic dependent launch (lei_apply_overlap, run concurrently with that
pass), and replays the whole step from a CUDA graph.  Here a 3-layer step run
that way must leave every bias and every gradient bit-identical to the same
layers run one after the other (plain lei_apply after each layer).
"""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def test_overlapped_graphed_step_equals_serial_layers(qb):
    sys.path.insert(0, ROOT)
    import bench
    from exact_distributed_quantiles_gb300 import inputs
    dev = torch.device("cuda", 0)
    a = bench.FullStep(qb, inputs, dev, layers=3)
    b = bench.FullStep(qb, inputs, dev, layers=3)
    # a: the bench's schedule, captured once and replayed twice
    a.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            a.step()
    torch.cuda.current_stream().wait_stream(cs)
    graph.replay()
    graph.replay()
    # b: three steps of layers strictly one after the other
    for _ in range(3):
        for l in range(3):
            b.layer(l, join=True)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    assert torch.equal(a.bias.view(torch.int32), b.bias.view(torch.int32))
    assert torch.equal(a.grads.view(torch.int32), b.grads.view(torch.int32))
    assert int(a.hist_hi.abs().sum()) == 0 and int(a.hist_lo.abs().sum()) == 0
