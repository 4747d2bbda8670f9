"""Pins for the oracle's exact quantile balancing (CPU only).

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph: the hi-byte histogram locates the bin that holds the r-th
smallest BF16 margin, a lo-byte histogram inside that bin finishes the select,
and the two bytes give the exact pooled quantile, whatever the sharding.
"[Dev] Add global-batch quantile balancing", "Quantile estimator" and
"Implementation": the quantile is at k/E, the result is mean-centred, every
expert's histogram row holds the same total.
"""
import json
import os

import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hx(s):
    return int(s, 16)


def test_golden_hand_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "eqb_hand_example.json")))
    E, k = g["E"], g["k"]
    m = np.array(g["margins_by_expert"], np.float32).T.copy()  # [N, E]
    N = m.shape[0]
    R = orc.rank(N, E, k)
    assert R == g["R"]
    key = orc.keys(m)
    h_hi = orc.hist_hi(key)
    for j in range(E):
        want = np.zeros(256, np.int32)
        for b, c in g["hist_hi_nonzero"][j].items():
            want[_hx(b)] = c
        assert np.array_equal(h_hi[j], want)
    sel, r_lo = orc.select_hi(h_hi, R)
    assert sel.tolist() == [_hx(s) for s in g["sel"]]
    assert r_lo.tolist() == g["r_lo"]
    h_lo = orc.hist_lo(key, sel)
    for j in range(E):
        want = np.zeros(256, np.int32)
        for b, c in g["hist_lo_nonzero"][j].items():
            want[_hx(b)] = c
        assert np.array_equal(h_lo[j], want)
    lo = orc.select_lo(h_lo, r_lo)
    assert lo.tolist() == [_hx(s) for s in g["lo"]]
    qkey = orc.kth_key(key, R)
    assert np.array_equal(qkey, (sel << 8 | lo).astype(np.uint16))
    q = orc.key_decode_array(qkey)
    assert q.tolist() == g["quantile"]
    b = orc.center(q.astype(np.float64))
    assert b.view(np.uint32).tolist() == [_hx(s) for s in g["bias_out_f32_bits"]]


def _small_pooled(seed=11, n_micro=8, n_tokens=512, E=64, k=6):
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=E, k=k, n_micro=n_micro, n_tokens=n_tokens)
    bias, mbs = inputs.router_layer(w, seed)
    return w, bias.numpy(), [x.numpy() for x in mbs]


def test_quantile_equals_library_kthvalue(orc):
    w, bias, mbs = _small_pooled()
    res = orc.eqb_global_batch(mbs, bias, w.k)
    margins = np.concatenate([orc.route(x, bias, w.k, want=("margins",))["margins"] for x in mbs])
    mb = torch.from_numpy(margins).to(torch.bfloat16).float()
    kth = torch.kthvalue(mb, res["R"], dim=0).values.numpy()
    assert np.array_equal(res["q"].astype(np.float32), kth)


def test_quantile_brute_force_definition(orc):
    rng = np.random.default_rng(5)
    N, E, k = 40, 8, 2
    logits = rng.normal(size=(N, E)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    res = orc.eqb_global_batch([logits], bias, k)
    m = orc.route(logits, bias, k, want=("margins",))["margins"]
    vals = orc.key_decode_array(orc.keys(m)).astype(np.float64)  # BF16-rounded margins
    R = -((-k * N) // E)
    for j in range(E):
        col = vals[:, j]
        cands = [x for x in col if np.sum(col <= x) >= R > np.sum(col < x)]
        assert len(set(cands)) == 1
        assert res["q"][j] == cands[0]


def test_invariants(orc):
    w, bias, mbs = _small_pooled(seed=12)
    res = orc.eqb_global_batch(mbs, bias, w.k)
    n_pool = w.n_pool
    # every expert row of the hi histogram holds the pooled token count
    assert np.all(res["hist_hi"].sum(axis=1) == n_pool)
    # the lo histogram holds exactly the samples of the selected hi bin
    sel = res["sel"]
    assert np.array_equal(res["hist_lo"].sum(axis=1), res["hist_hi"][np.arange(w.E), sel])
    # rank conditions on the keys: #{key <= q} >= R > #{key < q}
    allk = np.concatenate(res["keys"]).astype(np.int64)
    qk = res["qkey"].astype(np.int64)
    assert np.all((allk <= qk).sum(axis=0) >= res["R"])
    assert np.all((allk < qk).sum(axis=0) < res["R"])
    # centred: the new biases sum to zero up to their fp32 rounding
    b = res["bias_out"].astype(np.float64)
    assert abs(b.sum()) <= w.E * 2.0 ** -24 * np.abs(b).max()
    assert np.all(b == res["bias_out"])


@pytest.mark.parametrize("splits", [(2, 2048), (32, 128), (1, 4096)])
def test_partition_invariance(orc, splits):
    w, bias, mbs = _small_pooled(seed=13, n_micro=8, n_tokens=512)
    base = orc.eqb_global_batch(mbs, bias, w.k)
    allx = np.concatenate(mbs)
    n_m, n_t = splits
    parts = [allx[i * n_t:(i + 1) * n_t] for i in range(n_m)]
    other = orc.eqb_global_batch(parts, bias, w.k)
    for key in ("hist_hi", "hist_lo", "sel", "r_lo", "qkey", "bias_out"):
        assert np.array_equal(base[key], other[key]), key


def test_rank_local_histograms_differ(orc):
    # Pre-reduction histograms of different microbatches are not identical;
    # only their sum is what the quantile is read from.
    w, bias, mbs = _small_pooled(seed=14, n_micro=4, n_tokens=512)
    res = orc.eqb_global_batch(mbs, bias, w.k)
    locals_ = [orc.hist_hi(kk) for kk in res["keys"]]
    assert not np.array_equal(locals_[0], locals_[1])
    assert np.array_equal(sum(locals_), res["hist_hi"])


def test_bias_update_balances_the_batch(orc):
    # Informative: routing the same batch with the new bias moves every
    # expert's load towards N*k/E (alpha shifts with b, so not exact).
    w, bias, mbs = _small_pooled(seed=15, n_micro=4, n_tokens=1024)
    res = orc.eqb_global_batch(mbs, bias, w.k)
    allx = np.concatenate(mbs)

    def maxvio(b):
        t = orc.route(allx, b, w.k, want=("topk",))["topk"]
        load = np.bincount(t.ravel(), minlength=w.E)
        mean = t.size / w.E
        return (load.max() - mean) / mean

    assert maxvio(res["bias_out"]) < 0.5 * maxvio(bias)
