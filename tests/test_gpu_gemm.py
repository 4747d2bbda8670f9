"""Router GEMM on the tensor cores (tcgen05) and the router-GEMM workload.

The GEMM is checked against an fp64 product within the fp32 accumulation
error bound |err| <= 2 * H * 2^-24 * sum_k |h_k w_k| (per output); the EQB hi
pass run on the GEMM's own fp32 logits is checked bit for bit against the
oracle fed the same logits ("[Dev] Add global-batch quantile balancing",
"Implementation": the histogram pass extends the router kernel).
"""
import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs
from qb_testlib import assert_route_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _check_gemm(logits, hidden, W):
    h64 = hidden.double()
    w64 = W.double()
    exact = h64 @ w64
    bound = 2.0 * hidden.shape[1] * 2.0 ** -24 * (h64.abs() @ w64.abs()) + 1e-30
    err = (logits.double() - exact).abs()
    assert bool((err <= bound).all()), float((err / bound).max())
    return exact


@pytest.mark.parametrize("M,H,E", [(128, 64, 256), (300, 128, 256), (1000, 2048, 256),
                                   (129, 1024, 256), (1000, 512, 32), (333, 256, 96),
                                   (700, 2048, 160), (257, 128, 224)])
def test_router_gemm_small(qb, M, H, E):
    g = torch.Generator(device="cuda")
    g.manual_seed(M + H + E)
    hidden = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(H, E, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    w_t = W.t().contiguous()
    logits = torch.full((M, E), float("nan"), dtype=torch.float32, device="cuda")
    qb.qb_router_gemm(hidden, w_t, logits)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    assert torch.isfinite(logits).all()
    _check_gemm(logits, hidden, W)


def test_router_gemm_workload(qb, orc):
    # one microbatch of the router-GEMM workload: hidden [32768, 2048] bf16,
    # W [2048, 256] bf16 (variance 1/2048), k = 6
    w = inputs.WORKLOADS["router_gemm"]
    bias, W, hs = inputs.gemm_layer(inputs.scaled(w, n_micro=1), inputs.seed_for("router_gemm"),
                                    device="cuda")
    hidden = hs[0]
    w_t = W.t().contiguous()
    logits = torch.empty(w.n_tokens, w.E, dtype=torch.float32, device="cuda")
    hist = torch.zeros(w.E, 256, dtype=torch.int32, device="cuda")
    keys = torch.empty(w.n_tokens, w.E, dtype=torch.int16, device="cuda")
    topk = torch.empty(w.n_tokens, w.k, dtype=torch.int32, device="cuda")
    alpha = torch.empty(w.n_tokens, dtype=torch.float32, device="cuda")
    qb.qb_router_gemm_hist_hi(hidden, w_t, bias, w.k, logits, hist, keys_out=keys, topk_out=topk,
                              alpha_out=alpha)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    rows = torch.randperm(w.n_tokens, device="cuda")[:2048]
    _check_gemm(logits[rows], hidden[rows], W)
    res = dict(alpha=alpha.cpu().numpy(), keys=keys.cpu().numpy().view(np.uint16),
               topk=topk.cpu().numpy())
    ref = assert_route_matches(orc, res, logits.cpu().numpy(), bias.cpu().numpy(), w.k)
    assert np.array_equal(hist.cpu().numpy(), orc.hist_hi(orc.keys(ref["margins"])))


def _fused(qb, hidden, w_t, bias, k, with_logits=True):
    M = hidden.shape[0]
    dev = hidden.device
    logits = torch.empty(M, 256, dtype=torch.float32, device=dev) if with_logits else None
    hist = torch.zeros(256, 256, dtype=torch.int32, device=dev)
    keys = torch.empty(M, 256, dtype=torch.int16, device=dev)
    topk = torch.empty(M, k, dtype=torch.int32, device=dev)
    alpha = torch.empty(M, dtype=torch.float32, device=dev)
    qb.qb_router_gemm_hist_hi(hidden, w_t, bias, k, logits, hist, keys_out=keys, topk_out=topk,
                              alpha_out=alpha)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    return logits, dict(hist=hist.cpu().numpy(), keys=keys.cpu().numpy().view(np.uint16),
                        topk=topk.cpu().numpy(), alpha=alpha.cpu().numpy())


@pytest.mark.parametrize("M,H,k", [(1000, 128, 6), (300, 2048, 8), (129, 64, 1), (5000, 256, 15)])
def test_fused_epilogue_matches_routing_of_its_logits(qb, orc, M, H, k):
    g = torch.Generator(device="cuda")
    g.manual_seed(M * 7 + H + k)
    hidden = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(H, 256, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    w_t = W.t().contiguous()
    bias = (torch.rand(256, generator=g, device="cuda") * 2 - 1) * 0.1
    logits, res = _fused(qb, hidden, w_t, bias, k)
    # the epilogue's logits are the plain GEMM's, bit for bit (same MMA sequence)
    plain = torch.empty_like(logits)
    qb.qb_router_gemm(hidden, w_t, plain)
    torch.cuda.synchronize()
    assert torch.equal(logits.view(torch.int32), plain.view(torch.int32))
    ref = assert_route_matches(orc, res, logits.cpu().numpy(), bias.cpu().numpy(), k)
    assert np.array_equal(res["hist"], orc.hist_hi(orc.keys(ref["margins"])))
    # without logits_out the outputs are the same
    _, res2 = _fused(qb, hidden, w_t, bias, k, with_logits=False)
    for key in ("hist", "keys", "topk", "alpha"):
        assert np.array_equal(res2[key], res[key]), key


@pytest.mark.parametrize("M,H,E,k", [(700, 256, 96, 6), (300, 512, 160, 8), (129, 64, 32, 1)])
def test_fused_entry_other_expert_counts(qb, orc, M, H, E, k):
    # E != 256: the GEMM into logits_out, then the routing pass on it; the
    # same outputs as the routing pass on those logits, and no logits_out
    # is refused
    g = torch.Generator(device="cuda")
    g.manual_seed(M + H + E + k)
    hidden = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(H, E, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    w_t = W.t().contiguous()
    bias = (torch.rand(E, generator=g, device="cuda") * 2 - 1) * 0.1
    logits = torch.empty(M, E, dtype=torch.float32, device="cuda")
    hist = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    keys = torch.empty(M, E, dtype=torch.int16, device="cuda")
    topk = torch.empty(M, k, dtype=torch.int32, device="cuda")
    alpha = torch.empty(M, dtype=torch.float32, device="cuda")
    qb.qb_router_gemm_hist_hi(hidden, w_t, bias, k, logits, hist, keys_out=keys, topk_out=topk,
                              alpha_out=alpha)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    _check_gemm(logits, hidden, W)
    res = dict(hist=hist.cpu().numpy(), keys=keys.cpu().numpy().view(np.uint16),
               topk=topk.cpu().numpy(), alpha=alpha.cpu().numpy())
    ref = assert_route_matches(orc, res, logits.cpu().numpy(), bias.cpu().numpy(), k)
    assert np.array_equal(res["hist"], orc.hist_hi(orc.keys(ref["margins"])))
    with pytest.raises(qb.QBError):
        qb.qb_router_gemm_hist_hi(hidden, w_t, bias, k, None, hist)


def test_fused_epilogue_exact_path_on_ties(qb, orc):
    # W's 256 columns repeat 8 distinct ones: every group of 8 experts holds
    # the same values, so all 32 groups tie at tau (more candidates than the
    # staging holds) and alpha is tied many times over; bias 0
    M, H, k = 512, 128, 6
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    hidden = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W8 = (torch.randn(H, 8, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    W = W8.repeat(1, 32)
    w_t = W.t().contiguous()
    bias = torch.zeros(256, dtype=torch.float32, device="cuda")
    logits, res = _fused(qb, hidden, w_t, bias, k)
    ref = assert_route_matches(orc, res, logits.cpu().numpy(), bias.cpu().numpy(), k)
    assert np.array_equal(res["hist"], orc.hist_hi(orc.keys(ref["margins"])))


def test_fused_counts_past_one_launch(qb):
    # More tokens than one launch of the fused kernel covers (SMs x 511 tiles
    # x 128 tokens): the call is split so that no CTA's 16-bit window counter
    # sees 2^16 tokens.  The first half of the hidden rows are identical, so
    # every token of a CTA there lands in the same bin of each expert and an
    # overflowing counter would show; the counts and keys must equal those of
    # the plain GEMM followed by the routing kernel (32-bit counters).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, H, E, k = sms * 511 * 128 + 1037, 64, 256, 6
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    hidden = torch.randn(1, H, generator=g, device="cuda").expand(M, H).contiguous()
    hidden[M // 2:] = torch.randn(M - M // 2, H, generator=g, device="cuda")
    hidden = hidden.to(torch.bfloat16)
    w_t = (torch.randn(E, H, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    bias = (torch.rand(E, generator=g, device="cuda") * 2 - 1) * 0.1
    hist_f = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    keys_f = torch.empty(M, E, dtype=torch.int16, device="cuda")
    qb.qb_router_gemm_hist_hi(hidden, w_t, bias, k, None, hist_f, keys_out=keys_f)
    logits = torch.empty(M, E, dtype=torch.float32, device="cuda")
    qb.qb_router_gemm(hidden, w_t, logits)
    hist_r = torch.zeros_like(hist_f)
    keys_r = torch.empty_like(keys_f)
    qb.qb_route_hist_hi(logits, bias, k, hist_r, keys_out=keys_r)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    assert int(hist_f.sum()) == M * E
    assert int(hist_f.max()) >= 1 << 16  # some bin holds more than a 16-bit counter can
    assert torch.equal(hist_f, hist_r)
    assert torch.equal(keys_f, keys_r)


@pytest.mark.parametrize("chained", [False, True])
def test_router_gemm_global_batch_chain(qb, orc, chained):
    # The router-GEMM workload end to end: four 32768-token microbatches of
    # the fused GEMM + hi pass (logits kept in tensor memory), then select,
    # the lo pass over the stored keys and the finalize.  Histograms, selected
    # bins and keys, and the new bias are compared bit for bit with the oracle
    # fed the plain GEMM's fp32 logits, which equal the fused kernel's bit for
    # bit (test_fused_epilogue_matches_routing_of_its_logits).  chained: the
    # microbatches after the first through qb_router_gemm_hist_hi_next.
    w = inputs.WORKLOADS["router_gemm"]
    bias, W, hs = inputs.gemm_layer(w, inputs.seed_for("router_gemm"), device="cuda")
    w_t = W.t().contiguous()
    n, E = w.n_tokens, w.E
    st = qb.EQBState(E, "cuda")
    keys = torch.empty(w.n_pool, E, dtype=torch.int16, device="cuda")
    for i, h in enumerate(hs):
        f = qb.qb_router_gemm_hist_hi_next if chained and i else qb.qb_router_gemm_hist_hi
        f(h, w_t, bias, w.k, None, st.hist_hi, keys_out=keys[i * n:(i + 1) * n])
    hist_hi = st.hist_hi.clone()
    qb.qb_select_hi(st.hist_hi, qb.rank(w.n_pool, E, w.k), st.sel, st.r_lo)
    qb.qb_keys_hist_lo(keys, st.sel, st.hist_lo)
    hist_lo = st.hist_lo.clone()
    b_out = torch.empty_like(bias)
    qb.qb_finalize(st.hist_hi, st.hist_lo, st.sel, st.r_lo, b_out, qkey_out=st.qkey, reset=True)
    logits = []
    for h in hs:
        lg = torch.empty(n, E, dtype=torch.float32, device="cuda")
        qb.qb_router_gemm(h, w_t, lg)
        logits.append(lg)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    ref = orc.eqb_global_batch([lg.cpu().numpy() for lg in logits], bias.cpu().numpy(), w.k)
    assert np.array_equal(hist_hi.cpu().numpy(), ref["hist_hi"])
    assert np.array_equal(hist_lo.cpu().numpy(), ref["hist_lo"])
    assert np.array_equal(st.sel.cpu().numpy(), ref["sel"])
    assert np.array_equal(st.qkey.cpu().numpy().view(np.uint16), ref["qkey"])
    assert np.array_equal(b_out.cpu().numpy().view(np.uint32), ref["bias_out"].view(np.uint32))
    assert int(st.hist_hi.abs().sum()) == 0 and int(st.hist_lo.abs().sum()) == 0  # reset
