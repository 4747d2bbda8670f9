"""The library's calls inside a CUDA graph.

Every entry point is asynchronous on the caller's stream, allocates nothing
and keeps no per-call host state, so a layer's whole EQB + LEI sequence can
be captured once and replayed ("[Dev] Add global-batch quantile balancing",
"Implementation": persistent histogram and bias addresses, in-place update
and reset, so the same buffers serve every global batch).
"""
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


def test_layer_replayed_from_a_graph_equals_direct_calls(qb):
    w = inputs.scaled(inputs.WORKLOADS["full_step"], n_micro=4)
    n, E, k = w.n_pool, w.E, w.k
    logits = torch.empty(n, E, dtype=torch.float32, device="cuda")
    bias0, _ = inputs.router_layer(w, inputs.seed_for("full_step", 3), device="cuda", out=logits)
    grad0 = inputs.score_grad(w, inputs.seed_for("full_step", 3), n_tokens=n, device="cuda")
    bias = bias0.clone()
    grad = grad0.clone()
    hi = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    lo = torch.zeros_like(hi)
    sel = torch.empty(E, dtype=torch.int32, device="cuda")
    r_lo = torch.empty_like(sel)
    keys = torch.empty(n, E, dtype=torch.int16, device="cuda")
    topk = torch.empty(n, k, dtype=torch.int32, device="cuda")
    ws = torch.empty(w.n_micro, E, dtype=torch.float32, device="cuda")
    R = qb.rank(n, E, k)

    def layer():
        qb.qb_route_hist_hi(logits, bias, k, hi, keys_out=keys, topk_out=topk)
        qb.qb_select_hi(hi, R, sel, r_lo)
        qb.qb_keys_hist_lo(keys, sel, lo)
        qb.qb_finalize(hi, lo, sel, r_lo, bias, reset=True)
        qb.lei_inject(grad, topk, w.eta, ws, batch_tokens=w.n_tokens)

    layer()  # direct, on the current stream (also sets the kernels' attributes)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    bias_direct, grad_direct = bias.clone(), grad.clone()

    bias.copy_(bias0)
    grad.copy_(grad0)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # capture did not run anything: the buffers still hold the initial state
    assert torch.equal(bias, bias0) and int(hi.abs().sum()) == 0
    graph.replay()
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    assert torch.equal(bias.view(torch.int32), bias_direct.view(torch.int32))
    assert torch.equal(grad.view(torch.int32), grad_direct.view(torch.int32))
    assert int(hi.abs().sum()) == 0 and int(lo.abs().sum()) == 0  # reset in place


def test_chained_microbatch_calls_replayed_from_a_graph(qb):
    # The microbatch calls after the first are qb_route_hist_hi_next, whose
    # programmatic dependencies become graph edges; three replays of the
    # captured global batch (each routing with the bias the one before wrote)
    # equal three direct runs.
    w = inputs.scaled(inputs.WORKLOADS["full_step"], n_micro=8, n_tokens=8192)
    n, E, k = w.n_pool, w.E, w.k
    logits = torch.empty(n, E, dtype=torch.float32, device="cuda")
    bias0, mbs = inputs.router_layer(w, inputs.seed_for("full_step", 5), device="cuda",
                                     out=logits)
    bias = bias0.clone()
    hi = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    lo = torch.zeros_like(hi)
    sel = torch.empty(E, dtype=torch.int32, device="cuda")
    r_lo = torch.empty_like(sel)
    keys = torch.empty(n, E, dtype=torch.int16, device="cuda")
    R = qb.rank(n, E, k)

    def batch():
        for m, x in enumerate(mbs):
            route = qb.qb_route_hist_hi if m == 0 else qb.qb_route_hist_hi_next
            route(x, bias, k, hi, keys_out=keys[m * w.n_tokens:(m + 1) * w.n_tokens])
        qb.qb_select_hi(hi, R, sel, r_lo)
        qb.qb_keys_hist_lo(keys, sel, lo)
        qb.qb_finalize(hi, lo, sel, r_lo, bias, reset=True)

    direct = []
    for _ in range(3):
        batch()
        direct.append(bias.clone())
    torch.cuda.synchronize()
    assert qb.device_status() == 0

    bias.copy_(bias0)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            batch()
    torch.cuda.current_stream().wait_stream(s)
    for step in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(bias.view(torch.int32), direct[step].view(torch.int32)), step
    assert qb.device_status() == 0
    assert int(hi.abs().sum()) == 0 and int(lo.abs().sum()) == 0
