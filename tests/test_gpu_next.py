"""GPU parity of rank-averaged QB and MaxVio against the oracle (bit-exact).

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts":
opening paragraph (rank-averaged quantiles depend on the sharding) and testbed
paragraph (MaxVio, global and local).
"""
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


def _rank_qkeys(qb, rank_mbs, bias, k):
    """Each rank's EQB on its own tokens; returns the selected keys [P, E]."""
    E = bias.shape[0]
    qk = torch.empty(len(rank_mbs), E, dtype=torch.int16, device="cuda")
    for p, mbs in enumerate(rank_mbs):
        n = sum(int(m.shape[0]) for m in mbs)
        keys = torch.empty(n, E, dtype=torch.int16, device="cuda")
        hi = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
        lo = torch.zeros_like(hi)
        row = 0
        for m in mbs:
            qb.qb_route_hist_hi(m, bias, k, hi, keys_out=keys[row:row + m.shape[0]])
            row += m.shape[0]
        sel = torch.empty(E, dtype=torch.int32, device="cuda")
        r_lo = torch.empty_like(sel)
        qb.qb_select_hi(hi, qb.rank(n, E, k), sel, r_lo)
        qb.qb_keys_hist_lo(keys, sel, lo)
        scratch = torch.empty(E, dtype=torch.float32, device="cuda")
        qb.qb_finalize(hi, lo, sel, r_lo, scratch, qkey_out=qk[p], reset=True)
    return qk


@pytest.mark.parametrize("shards", [1, 2, 8])
def test_rank_average_pooled_workload(qb, orc, shards):
    # the pooled workload (8 skewed microbatches of 16384) as `shards` ranks
    w = inputs.WORKLOADS["eqb_pooled"]
    bias, mbs = inputs.router_layer(w, inputs.seed_for("eqb_pooled"), device="cuda")
    per = len(mbs) // shards
    rank_mbs = [mbs[p * per:(p + 1) * per] for p in range(shards)]
    qk = _rank_qkeys(qb, rank_mbs, bias, w.k)
    out = torch.empty_like(bias)
    qb.qb_rank_average(qk, out)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    ref = orc.rank_averaged_qb([[m.cpu().numpy() for m in r] for r in rank_mbs],
                               bias.cpu().numpy(), w.k)
    assert np.array_equal(qk.cpu().numpy().view(np.uint16), ref["qkey_rank"])
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref["bias_out"].view(np.uint32))


@pytest.mark.parametrize("N,E,k,bt", [(131072, 256, 6, 32768), (1000, 64, 6, 333),
                                      (4097, 512, 15, 1024), (77, 32, 1, 0),
                                      (3001, 1024, 8, 1000), (2000, 352, 6, 640)])
def test_maxvio(qb, orc, N, E, k, bt):
    topk = inputs.random_topk(N, E, k, seed=N + E, device="cuda")
    topk[: N // 5] = torch.arange(k, dtype=torch.int32, device="cuda")  # a hot set of experts
    nb = 1 if bt == 0 else (N + bt - 1) // bt
    loads = torch.full((nb, E), -1, dtype=torch.int32, device="cuda")
    mv = torch.empty(2, dtype=torch.float64, device="cuda")
    qb.qb_maxvio(topk, E, loads, mv, batch_tokens=bt)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    t = topk.cpu().numpy()
    step = N if bt == 0 else bt
    ref = orc.maxvio([t[i:i + step] for i in range(0, N, step)], E)
    assert np.array_equal(loads.cpu().numpy(), ref["loads"])
    got = mv.cpu().numpy()
    assert got[0] == ref["global_maxvio"] and got[1] == ref["local_maxvio"]
