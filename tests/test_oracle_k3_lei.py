"""Pins for the oracle's K3 histogram quantile and LEI (CPU only).

K3: "[Dev] Add global-batch quantile balancing", "Quantile estimator" (uniform
bins per expert over [min(b)-1, max(b)+1]) and "Implementation" (one int32
histogram per router pooled over every microbatch); its accuracy is capped by
the bin width ("Exact Quantile Balancing ...", paragraph on K3's histogram).
LEI: "Exact Quantile Balancing and Load-Error Injection for Mixture-of-
Experts", LEI paragraph.
"""
import json
import os

import numpy as np
import pytest

from exact_distributed_quantiles_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ K3

def test_k3_golden_hand_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "k3_hand_example.json")))
    m = np.array(g["margins_by_expert"], np.float32).T.copy()
    R = orc.rank(m.shape[0], g["E"], g["k"])
    assert R == g["R"]
    h = orc.k3_hist(m, g["lo"], g["hi"], g["nbins"])
    assert h.tolist() == g["hist"]
    b, bounds, q = orc.k3_finalize(h, R, g["lo"], g["hi"])
    assert np.allclose(q, g["quantile"], rtol=0, atol=1e-15)
    assert np.array_equal(b, np.float32(g["bias_out"]))
    assert np.array_equal(bounds, np.float32(g["bounds_out"]))


def test_k3_clamps_out_of_range_margins(orc):
    m = np.float32([[-3.0], [-1.0], [0.99], [1.0], [7.0], [-1.0000001]])
    h = orc.k3_hist(m, -1.0, 1.0, 4)
    # below lo -> bin 0; lo itself -> bin 0; hi and above -> last bin
    assert h.tolist() == [[3, 0, 0, 3]]


def _k3_small(seed=21, n_micro=4, n_tokens=512, E=64, k=8, nbins=1000):
    w = inputs.scaled(inputs.WORKLOADS["k3"], E=E, k=k, n_micro=n_micro, n_tokens=n_tokens, nbins=nbins)
    bias, mbs = inputs.router_layer(w, seed)
    bounds = inputs.k3_initial_bounds(bias).numpy()
    bits = [x.view(__import__("torch").int16).numpy().view(np.uint16) for x in mbs]
    return w, bias.numpy(), bits, bounds


def test_k3_within_one_bin_of_exact_quantile(orc):
    w, bias, mbs, bounds = _k3_small()
    res = orc.k3_global_batch(mbs, bias, w.k, bounds, w.nbins)
    margins = np.concatenate([orc.route(x, bias, w.k, want=("margins",))["margins"] for x in mbs])
    exact = np.sort(margins.astype(np.float64), axis=0)[res["R"] - 1]
    width = (float(bounds[1]) - float(bounds[0])) / w.nbins
    assert np.all(np.abs(res["q"] - exact) <= width * (1 + 1e-5))
    # and strictly better than a coarse histogram would promise
    assert np.mean(np.abs(res["q"] - exact)) < 0.5 * width


def test_k3_range_holds_every_margin(orc):
    # With the bias that defines [min b - 1, max b + 1], each margin
    # alpha - s_j lies strictly inside: alpha > min b (s > 0) and s_j < 1.
    w, bias, mbs, bounds = _k3_small(seed=22)
    lo, hi = np.float32(bounds[0]), np.float32(bounds[1])
    for x in mbs:
        m = orc.route(x, bias, w.k, want=("margins",))["margins"]
        assert np.all(m > lo) and np.all(m < hi)


def test_k3_invariants_and_partition(orc):
    w, bias, mbs, bounds = _k3_small(seed=23)
    res = orc.k3_global_batch(mbs, bias, w.k, bounds, w.nbins)
    assert np.all(res["hist"].sum(axis=1) == w.n_pool)
    b = res["bias_out"].astype(np.float64)
    assert abs(b.sum()) <= w.E * 2.0 ** -24 * np.abs(b).max()
    assert res["bounds_out"][0] == np.float32(res["bias_out"].min() - np.float32(1.0))
    assert res["bounds_out"][1] == np.float32(res["bias_out"].max() + np.float32(1.0))
    allx = np.concatenate(mbs)
    other = orc.k3_global_batch([allx[:300], allx[300:]], bias, w.k, bounds, w.nbins)
    assert np.array_equal(res["hist"], other["hist"])
    assert np.array_equal(res["bias_out"], other["bias_out"])


# ------------------------------------------------------------------ LEI

def test_lei_golden_hand_example(orc):
    g = json.load(open(os.path.join(GOLDEN, "lei_hand_example.json")))
    E = g["E"]
    topk = np.array(g["topk"], np.int32)
    grad = np.zeros((topk.shape[0], E), np.float32)
    new, load, rho = orc.lei(grad, topk, g["eta"])
    assert load.tolist() == g["load"]
    assert np.allclose(rho, g["rho"], rtol=0, atol=1e-15)
    c = (np.float64(np.float32(g["eta"])) * np.array(g["rho"])).astype(np.float32)
    assert np.array_equal(new, np.broadcast_to(c, new.shape))


def test_lei_uniform_load_leaves_gradient_unchanged(orc):
    N, k, E = 64, 4, 16
    # token i picks experts (4i .. 4i+3) mod 16: every expert gets N*k/E
    topk = (np.arange(N)[:, None] * k + np.arange(k)[None, :]) % E
    rng = np.random.default_rng(0)
    grad = rng.normal(0, 1e-3, size=(N, E)).astype(np.float32)
    new, load, rho = orc.lei(grad, topk.astype(np.int32), 8e-5)
    assert np.all(load == N * k // E)
    assert np.all(rho == 0.0)
    assert np.array_equal(new, grad)


def test_lei_properties(orc):
    N, E, k = 2048, 64, 6
    topk = inputs.random_topk(N, E, k, seed=3).numpy()
    # skew: send a block of tokens to experts 0..5 to create real imbalance
    topk[:300] = np.arange(6)[None, :]
    rng = np.random.default_rng(1)
    grad = rng.normal(0, 1e-3, size=(N, E)).astype(np.float32)
    eta = 8e-5
    new, load, rho = orc.lei(grad, topk, eta)
    assert load.sum() == N * k
    # zero-centred and bounded (tanh in (-1, 1), minus its mean)
    assert abs(rho.sum()) < 1e-12
    assert np.all(np.abs(rho) < 2.0)
    # direction kept: more load -> larger rho (tanh is monotone, centring is a shift)
    order = np.argsort(load, kind="stable")
    assert np.all(np.diff(rho[order]) >= 0)
    assert np.all((np.diff(load[order]) > 0) <= (np.diff(rho[order]) > 0))
    # the most loaded expert is pushed down by descent, the least loaded pulled up
    assert rho[np.argmax(load)] > 0 and rho[np.argmin(load)] < 0
    # every token of the local batch receives the same per-expert correction
    delta = new.astype(np.float64) - grad.astype(np.float64)
    c = eta * rho
    assert np.all(np.abs(delta - c[None, :]) <= np.spacing(np.abs(new)).astype(np.float64)
                  + np.spacing(np.float32(np.abs(c).max())))
