"""GPU parity of the K3 histogram path, LEI and the pinned logistic function.

K3: "[Dev] Add global-batch quantile balancing", "Quantile estimator" and
"Implementation" -- counts exact, biases within 1e-6 relative to the scale of
the centering, max(max_j |b_j|, max_j |q_j|) over the oracle's biases b and
uncentered quantiles q (the GPU sums the fp64 quantiles in a fixed tree, the
oracle in ascending order, so when every b_j is ~0 -- all quantiles equal --
they differ at the rounding of the q_j, not of the b_j), and within the
device's rounding model below.
LEI: "Exact Quantile Balancing and Load-Error Injection for Mixture-of-
Experts", LEI paragraph -- gradients within 1e-6 absolute.
Sigmoid: the score function, bit-equal to the oracle over all 2^32 inputs.
"""
import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs
from qb_testlib import host_logits

pytestmark = pytest.mark.gpu

K3_REL_TOL = 1e-6
LEI_ABS_TOL = 1e-6


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


# ------------------------------------------------------------------ sigmoid

def test_sigmoid_bit_equal_on_every_binary32_input(qb, orc):
    chunk = 1 << 28
    # both device sequences: the packed fast path (with its per-chunk switch
    # to the scalar one for large inputs) and the scalar one on every input
    x = torch.empty(chunk, dtype=torch.float32, device="cuda")
    s = torch.empty_like(x)
    s1 = torch.empty_like(x)
    base = torch.arange(chunk, dtype=torch.int64, device="cuda")
    mism = mism_scalar = 0
    for c in range(1 << 4):
        bits = (base + c * chunk).to(torch.int64)
        bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits).to(torch.int32)
        x.copy_(bits.view(torch.float32))
        qb.qb_sigmoid(x, s)
        qb.qb_sigmoid_scalar(x, s1)
        xs = x.cpu().numpy()
        got = s.cpu().numpy().view(np.uint32)
        got1 = s1.cpu().numpy().view(np.uint32)
        want = orc.sigmoid(xs).view(np.uint32)
        fin = ~np.isnan(xs)
        mism += int(np.count_nonzero(got[fin] != want[fin]))
        mism_scalar += int(np.count_nonzero(got1[fin] != want[fin]))
    assert mism == 0
    assert mism_scalar == 0


# ------------------------------------------------------------------ K3

def _k3_gpu(qb, mbs, bias, k, bounds0, nbins, chained=False):
    # chained: the microbatches after the first through k3_route_hist_next,
    # with two alpha buffers used in turn
    E = bias.shape[0]
    hist = torch.zeros(E, nbins, dtype=torch.int32, device="cuda")
    bounds = bounds0.clone().cuda()
    alpha = torch.empty(2, max(m.shape[0] for m in mbs), dtype=torch.float32, device="cuda")
    for i, m in enumerate(mbs):
        route = qb.k3_route_hist_next if chained and i else qb.k3_route_hist
        route(m, bias, k, bounds, hist, alpha[i % 2, :m.shape[0]])
    n_pool = sum(m.shape[0] for m in mbs)
    h = hist.clone()
    b_out = torch.empty_like(bias)
    qb.k3_finalize(hist, qb.rank(n_pool, E, k), bounds, b_out, reset=True)
    torch.cuda.synchronize()
    assert int(hist.abs().sum()) == 0
    return h.cpu().numpy(), b_out.cpu().numpy(), bounds.cpu().numpy()


def _check_k3(res, ref, bounds0, nbins):
    h, b, bounds = res
    assert np.array_equal(h, ref["hist"])
    scale = max(float(np.abs(ref["bias_out"]).max()), float(np.abs(ref["q"]).max()))
    assert np.max(np.abs(b.astype(np.float64) - ref["bias_out"])) <= K3_REL_TOL * scale
    assert np.allclose(bounds, ref["bounds_out"], rtol=0, atol=K3_REL_TOL * scale)
    # Much tighter than the tolerance: the device differs from the oracle
    # only in rounding -- an fp32 in-bin fraction (relative error <= 2^-23,
    # scaled by the bin width), fp64 tree sums and reciprocal products, and
    # the final fp32 rounding of each bias (up to one ulp of it either way).
    lo, hi = (float(x) for x in np.asarray(bounds0, dtype=np.float64))
    width = (hi - lo) / nbins
    ulp = np.spacing(np.abs(ref["bias_out"]).astype(np.float32)).astype(np.float64)
    err = np.abs(b.astype(np.float64) - ref["bias_out"].astype(np.float64))
    assert np.all(err <= 2 * ulp + width * 2.0 ** -22)


@pytest.mark.parametrize("chained", [False, True])
def test_k3_workload(qb, orc, chained):
    w = inputs.WORKLOADS["k3"]
    bias, mbs = inputs.router_layer(w, inputs.seed_for("k3"), device="cuda")
    b0 = inputs.k3_initial_bounds(bias)
    res = _k3_gpu(qb, mbs, bias, w.k, b0, w.nbins, chained=chained)
    ref = orc.k3_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k,
                              b0.numpy(), w.nbins)
    _check_k3(res, ref, b0.numpy(), w.nbins)


@pytest.mark.parametrize("E,k,nbins,dtype", [(64, 6, 1000, torch.float32),
                                              (256, 8, 37, torch.bfloat16),
                                              (512, 15, 4096, torch.float32),
                                              (32, 1, 1000, torch.bfloat16),
                                              (128, 3, 1000, torch.float32),
                                              (64, 6, 8000, torch.float32),   # global counts
                                              (96, 6, 1000, torch.bfloat16),  # padded rows
                                              (384, 8, 1000, torch.float32),
                                              (1024, 8, 1000, torch.bfloat16),
                                              (32, 2, 1, torch.float32)])
def test_k3_small_shapes(qb, orc, E, k, nbins, dtype):
    w = inputs.scaled(inputs.WORKLOADS["k3"], E=E, k=k, n_micro=3, n_tokens=32 * 5 + 3,
                      nbins=nbins, logits_dtype=dtype)
    bias, mbs = inputs.router_layer(w, 31 + E, device="cuda")
    b0 = inputs.k3_initial_bounds(bias)
    res = _k3_gpu(qb, mbs, bias, w.k, b0, nbins, chained=E % 64 == 0)
    ref = orc.k3_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k,
                              b0.numpy(), nbins)
    _check_k3(res, ref, b0.numpy(), nbins)


def test_k3_out_of_range_clamps(qb, orc):
    # Narrow bounds that most margins fall outside: clamping to the edge bins.
    w = inputs.scaled(inputs.WORKLOADS["k3"], E=64, k=6, n_micro=1, n_tokens=500)
    bias, mbs = inputs.router_layer(w, 5, device="cuda")
    b0 = torch.tensor([-0.05, 0.05], dtype=torch.float32)
    res = _k3_gpu(qb, mbs, bias, w.k, b0, 100)
    ref = orc.k3_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k,
                              b0.numpy(), 100)
    assert ref["hist"][:, 0].sum() > 0 and ref["hist"][:, -1].sum() > 0
    _check_k3(res, ref, b0.numpy(), 100)


# ------------------------------------------------------------------ LEI

def test_lei_full_step_microbatches(qb, orc):
    # One layer of the full-step workload (16 local batches of 32768 tokens)
    # in the launch configuration the benchmark times: top-6 from the GPU hi
    # pass with the pre-update bias, lei_rho, then the grad update enqueued
    # behind the next layer's hi pass (lei_apply_overlap, running beside it);
    # eta = 8e-5, grad ~ N(0, 1e-3).  Every batch compared with the oracle.
    w = inputs.WORKLOADS["full_step"]
    out = torch.empty(w.n_pool, w.E, dtype=torch.float32, device="cuda")
    bias, _ = inputs.router_layer(w, inputs.seed_for("full_step", 1), device="cuda", out=out)
    topk = torch.empty(w.n_pool, w.k, dtype=torch.int32, device="cuda")
    keys = torch.empty(w.n_pool, w.E, dtype=torch.int16, device="cuda")
    hist = torch.zeros(w.E, 256, dtype=torch.int32, device="cuda")
    qb.qb_route_hist_hi(out, bias, w.k, hist, keys_out=keys, topk_out=topk)
    grad = inputs.score_grad(w, seed=1, n_tokens=w.n_pool, device="cuda")
    g0 = grad.cpu().numpy()
    ws = torch.empty(w.n_micro, w.E, dtype=torch.float32, device="cuda")
    qb.lei_rho(topk, w.E, w.eta, ws, batch_tokens=w.n_tokens)
    nxt = torch.empty_like(out)
    bias2, _ = inputs.router_layer(w, inputs.seed_for("full_step", 2), device="cuda", out=nxt)
    qb.qb_route_hist_hi(nxt, bias2, w.k, hist, keys_out=keys)  # the next layer's hi pass
    qb.lei_apply_overlap(grad, ws, batch_tokens=w.n_tokens)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    t = topk.cpu().numpy()
    got = grad.cpu().numpy()
    c_all = ws.cpu().numpy().astype(np.float64)
    for m in range(w.n_micro):
        sl = slice(m * w.n_tokens, (m + 1) * w.n_tokens)
        want, load, rho = orc.lei(g0[sl], t[sl], w.eta)
        assert load.sum() == w.n_tokens * w.k
        assert np.max(np.abs(got[sl] - want)) <= LEI_ABS_TOL
        # the workspace holds eta * rho; the device evaluates rho in fp32
        # (division, tanh and a 256-term mean: a few ulp of values <= 2), so
        # eta * rho is within eta * 2e-6 of the fp64 value
        assert np.max(np.abs(c_all[m] - w.eta * rho)) <= w.eta * 2e-6


@pytest.mark.parametrize("N,E,k,bt", [(1, 32, 1, 0), (1000, 64, 6, 333), (4097, 512, 15, 1024),
                                      (3001, 96, 6, 1000), (2049, 384, 8, 512)])
def test_lei_shapes_and_ragged_batches(qb, orc, N, E, k, bt):
    topk = inputs.random_topk(N, E, k, seed=N, device="cuda")
    topk[: N // 3] = torch.arange(k, dtype=torch.int32, device="cuda")  # imbalance
    g = torch.Generator(device="cuda")
    g.manual_seed(N)
    grad = torch.randn(N, E, generator=g, device="cuda") * 1e-3
    g0 = grad.cpu().numpy()
    bt_eff = bt or N
    nb = (N + bt_eff - 1) // bt_eff
    ws = torch.empty(nb, E, dtype=torch.float32, device="cuda")
    qb.lei_inject(grad, topk, 0.5, ws, batch_tokens=bt)
    torch.cuda.synchronize()
    t = topk.cpu().numpy()
    got = grad.cpu().numpy()
    for m in range(nb):
        sl = slice(m * bt_eff, min(N, (m + 1) * bt_eff))
        want, _, _ = orc.lei(g0[sl], t[sl], 0.5)
        assert np.max(np.abs(got[sl] - want)) <= LEI_ABS_TOL


@pytest.mark.parametrize("N,E,k,bt", [(1, 32, 1, 0), (1000, 64, 6, 333), (4097, 512, 15, 1024),
                                      (70001, 256, 6, 4099), (5003, 160, 6, 777),
                                      (4099, 480, 15, 1000), (2049, 1024, 8, 512)])
def test_lei_rho_then_apply_equals_inject(qb, orc, N, E, k, bt):
    # The two halves on one stream give lei_inject's result bit for bit;
    # lei_apply alone is grad + workspace[batch(row)] in binary32 for every
    # element, checked against numpy on the workspace it was given.  Batch
    # sizes that are not multiples of a CTA's rows put batch boundaries
    # inside a CTA's run.
    topk = inputs.random_topk(N, E, k, seed=N + 7, device="cuda")
    topk[: N // 4] = torch.arange(k, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(N + 7)
    grad = torch.randn(N, E, generator=g, device="cuda") * 1e-3
    g0 = grad.cpu().numpy()
    bt_eff = bt or N
    nb = (N + bt_eff - 1) // bt_eff
    ws_a = torch.empty(nb, E, dtype=torch.float32, device="cuda")
    ws_b = torch.empty_like(ws_a)
    grad_b = grad.clone()
    qb.lei_inject(grad, topk, 0.5, ws_a, batch_tokens=bt)
    qb.lei_rho(topk, E, 0.5, ws_b, batch_tokens=bt)
    qb.lei_apply(grad_b, ws_b, batch_tokens=bt)
    torch.cuda.synchronize()
    assert torch.equal(ws_a, ws_b)
    assert torch.equal(grad.view(torch.int32), grad_b.view(torch.int32))
    c = ws_b.cpu().numpy()
    rows = np.arange(N) // bt_eff
    want = (g0 + c[rows]).astype(np.float32)
    assert np.array_equal(grad_b.cpu().numpy().view(np.int32), want.view(np.int32))
    t = topk.cpu().numpy()
    got = grad_b.cpu().numpy()
    for m in range(nb):
        sl = slice(m * bt_eff, min(N, (m + 1) * bt_eff))
        want_m, _, _ = orc.lei(g0[sl], t[sl], 0.5)
        assert np.max(np.abs(got[sl] - want_m)) <= LEI_ABS_TOL


@pytest.mark.parametrize("N,E,bt", [(1, 32, 0), (1000, 64, 333), (4097, 512, 1024),
                                    (3001, 96, 1000), (2049, 384, 512), (1031, 1024, 300),
                                    (70001, 256, 4099), (524288, 256, 32768)])
def test_lei_apply_overlap_equals_apply(qb, N, E, bt):
    # The bulk-copy variant gives lei_apply's result bit for bit, alone and
    # launched behind a routing pass that it runs beside; the routing pass's
    # own outputs are unchanged by the kernel running next to it.
    g = torch.Generator(device="cuda")
    g.manual_seed(N + 11)
    grad = torch.randn(N, E, generator=g, device="cuda") * 1e-3
    bt_eff = bt or N
    nb = (N + bt_eff - 1) // bt_eff
    ws = torch.randn(nb, E, generator=g, device="cuda") * 1e-5
    # subnormal sums, signed zeros, exact cancellation and a large addend
    grad[0, :8] = torch.tensor([1e-39, -1e-39, 3e-45, 0.0, -0.0, 1e30, -2.0, 5e-38], device="cuda")
    ws[0, :8] = torch.tensor([0.0, 0.0, 0.0, -0.0, -0.0, 1.0, 2.0, -5e-38], device="cuda")
    want = grad.clone()
    qb.lei_apply(want, ws, batch_tokens=bt)
    g0 = grad.cpu().numpy()
    exact = (g0 + ws.cpu().numpy()[np.arange(N) // bt_eff]).astype(np.float32)
    assert np.array_equal(want.cpu().numpy().view(np.int32), exact.view(np.int32))
    alone = grad.clone()
    qb.lei_apply_overlap(alone, ws, batch_tokens=bt)
    torch.cuda.synchronize()
    assert torch.equal(alone.view(torch.int32), want.view(torch.int32))
    # behind a routing pass over other data
    w = inputs.scaled(inputs.WORKLOADS["full_step"], n_micro=2)
    lg = torch.empty(w.n_pool, w.E, dtype=torch.float32, device="cuda")
    bias, _ = inputs.router_layer(w, inputs.seed_for("full_step", 2), device="cuda", out=lg)
    outs = []
    for overlap in (False, True):
        hist = torch.zeros(w.E, 256, dtype=torch.int32, device="cuda")
        keys = torch.empty(w.n_pool, w.E, dtype=torch.int16, device="cuda")
        topk = torch.empty(w.n_pool, w.k, dtype=torch.int32, device="cuda")
        behind = grad.clone()
        torch.cuda.synchronize()
        qb.qb_route_hist_hi(lg, bias, w.k, hist, keys_out=keys, topk_out=topk)
        if overlap:
            qb.lei_apply_overlap(behind, ws, batch_tokens=bt)
            hist_after = hist.clone()  # ordered after both kernels
        torch.cuda.synchronize()
        outs.append((hist, keys, topk))
        if overlap:
            assert torch.equal(behind.view(torch.int32), want.view(torch.int32))
            assert torch.equal(hist_after, hist)
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    assert qb.device_status() == 0
