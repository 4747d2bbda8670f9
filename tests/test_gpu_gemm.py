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


@pytest.mark.parametrize("M,H", [(128, 64), (300, 128), (1000, 2048), (129, 1024)])
def test_router_gemm_small(qb, M, H):
    g = torch.Generator(device="cuda")
    g.manual_seed(M + H)
    hidden = torch.randn(M, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(H, 256, generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    w_t = W.t().contiguous()
    logits = torch.full((M, 256), float("nan"), dtype=torch.float32, device="cuda")
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
