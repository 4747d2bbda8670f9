"""Pins of the oracle's rank-averaged QB and MaxVio.

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts":
opening paragraph (the MARIN implementation averages rank-local quantiles,
so the result depends on the sharding) and testbed paragraph (MaxVio: how
far the busiest expert exceeds uniform load; global and local variants).
"""
import json
import os

import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_maxvio_hand_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "maxvio_hand_example.json")))
    res = orc.maxvio([np.array(t, np.int32) for t in g["topk_batches"]], g["E"])
    assert np.array_equal(res["loads"], np.array(g["loads"]))
    assert res["global_maxvio"] == g["global_maxvio"]
    assert res["local_maxvio"] == g["local_maxvio"]


def test_maxvio_closed_forms(orc):
    E, k = 16, 2
    # perfectly uniform assignment: every expert gets exactly T -> 0
    t = np.array([[(2 * i) % E, (2 * i + 1) % E] for i in range(64)], np.int32)
    r = orc.maxvio([t, t], E)
    assert r["global_maxvio"] == 0.0 and r["local_maxvio"] == 0.0
    # everything on two experts with k = 2: loads n, n -> (n - 2n/E)/(2n/E) = E/2 - 1
    t = np.tile(np.array([[3, 7]], np.int32), (40, 1))
    r = orc.maxvio([t], E)
    assert r["global_maxvio"] == E / 2 - 1 == r["local_maxvio"]
    # one batch: global and local agree
    rng = np.random.default_rng(0)
    t = np.argsort(rng.random((100, E)), axis=1)[:, :k].astype(np.int32)
    r = orc.maxvio([t], E)
    assert r["global_maxvio"] == r["local_maxvio"]


def _layer(E=64, n_micro=4, n_tokens=512, seed=77):
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=E, k=6, n_micro=n_micro, n_tokens=n_tokens)
    bias, mbs = inputs.router_layer(w, seed)
    return w, bias.numpy(), [m.numpy() for m in mbs]


def test_rank_average_one_rank_is_the_pooled_method(orc):
    w, b, mbs = _layer()
    ra = orc.rank_averaged_qb([mbs], b, w.k)
    eqb = orc.eqb_global_batch(mbs, b, w.k)
    assert np.array_equal(ra["bias_out"].view(np.uint32), eqb["bias_out"].view(np.uint32))


def test_rank_average_of_identical_ranks_is_the_pooled_method(orc):
    # P copies of the same shard: every rank has the same quantile, and when
    # k*N/E is an integer the pooled rank P*R picks the same key -> identical
    w, b, mbs = _layer(n_micro=2, n_tokens=512)
    assert (w.k * 2 * 512) % w.E == 0
    ra = orc.rank_averaged_qb([mbs, mbs, mbs], b, w.k)
    pooled = orc.eqb_global_batch(mbs * 3, b, w.k)
    assert np.array_equal(ra["bias_out"].view(np.uint32), pooled["bias_out"].view(np.uint32))
    assert np.array_equal(ra["q_rank"][0], ra["q_rank"][2])


def test_rank_average_depends_on_the_sharding(orc):
    # skewed microbatches: averaging rank quantiles is not the pooled quantile,
    # and two shardings of the same tokens disagree (the pooled method does not)
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=64, k=6, n_micro=4, n_tokens=1024)
    bias, mbs = inputs.router_layer(w, 5)
    b, mbs = bias.numpy(), [m.numpy() for m in mbs]
    by4 = orc.rank_averaged_qb([[m] for m in mbs], b, w.k)["bias_out"]
    by2 = orc.rank_averaged_qb([mbs[:2], mbs[2:]], b, w.k)["bias_out"]
    pooled = orc.eqb_global_batch(mbs, b, w.k)["bias_out"]
    assert not np.array_equal(by4, by2)
    assert not np.array_equal(by4, pooled)
    assert abs(float(by4.astype(np.float64).sum())) <= 64 * 2.0 ** -24 * float(np.abs(by4).max())
