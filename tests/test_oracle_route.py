"""Pins for the oracle's routing step (CPU only).

"[Dev] Add global-batch quantile balancing", "Quantile estimator": alpha[i] is
the (k+1)-th largest value of s[i,:] + b, and r[i,j] = alpha[i] - s[i,j].
Brute force over every element checks the definition; ties are planted on
purpose, because fp32 ties occur at 10^5 tokens x 256 experts.
"""
import numpy as np
import pytest


def _brute_alpha(v, k):
    # alpha is the value with fewer than k+1 elements above it and at least
    # k+1 elements at or above it.
    for cand in v:
        above = sum(1 for w in v if w > cand)
        at_or_above = sum(1 for w in v if w >= cand)
        if above < k + 1 <= at_or_above:
            return cand
    raise AssertionError("no alpha")


def _brute_topk(v, k):
    # Greedy: repeatedly take the largest remaining value, lowest index first.
    left = list(range(len(v)))
    out = []
    for _ in range(k):
        best = left[0]
        for j in left:
            if v[j] > v[best] or (v[j] == v[best] and j < best):
                best = j
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("E,k", [(8, 1), (8, 3), (16, 6), (7, 6)])
def test_route_brute_force_with_ties(orc, E, k):
    rng = np.random.default_rng(E * 100 + k)
    N = 60
    logits = rng.normal(size=(N, E)).astype(np.float32)
    # Plant exact ties in v: duplicate logits with equal bias entries.
    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    bias[1] = bias[0]
    bias[3] = bias[2]
    logits[::3, 1] = logits[::3, 0]
    logits[::2, 3] = logits[::2, 2]
    logits[::5, :] = logits[::5, :1]  # whole rows tied except for the bias ...
    bias_t = bias.copy()
    out = orc.route(logits, bias_t, k)
    s = orc.sigmoid(logits)
    assert np.array_equal(out["scores"], s)
    for i in range(N):
        v = [np.float32(s[i, j] + bias[j]) for j in range(E)]
        a = _brute_alpha(v, k)
        assert out["alpha"][i] == a
        assert out["topk"][i].tolist() == _brute_topk(v, k)
        m = (np.float32(a) - s[i]).astype(np.float32)
        assert np.array_equal(out["margins"][i], m)


def test_route_all_equal_row(orc):
    E, k = 8, 3
    logits = np.zeros((2, E), np.float32)
    bias = np.zeros(E, np.float32)
    out = orc.route(logits, bias, k)
    assert np.all(out["alpha"] == 0.5)
    assert np.all(out["margins"] == 0.0)
    assert out["topk"].tolist() == [[0, 1, 2], [0, 1, 2]]


def test_alpha_matches_partition(orc):
    rng = np.random.default_rng(3)
    N, E, k = 500, 64, 6
    logits = rng.normal(size=(N, E)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, size=E).astype(np.float32)
    out = orc.route(logits, bias, k)
    v = (orc.sigmoid(logits) + bias[None, :]).astype(np.float32)
    # (k+1)-th largest value = element E-1-k of an ascending partition
    ref = np.partition(v, E - 1 - k, axis=1)[:, E - 1 - k]
    assert np.array_equal(out["alpha"], ref)
    # Selection in margin form: expert j is among the top k exactly when
    # s_j + b_j >= alpha, i.e. r_j <= b_j (up to the rounding of v and r).
    m = out["margins"]
    tol = 2e-7
    for i in range(N):
        sel = out["topk"][i]
        assert np.all(m[i, sel] <= bias[sel] + tol)
        rest = np.setdiff1d(np.arange(E), sel)
        assert np.sum(m[i, rest] < bias[rest] - tol) == 0


def test_bf16_logits_route_like_upcast_fp32(orc):
    rng = np.random.default_rng(4)
    x = rng.normal(size=(64, 32)).astype(np.float32)
    import torch
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    bias = rng.uniform(-0.2, 0.2, size=32).astype(np.float32)
    a = orc.route(bits, bias, 8)
    b = orc.route(xb.float().numpy(), bias, 8)
    for key in a:
        assert np.array_equal(a[key], b[key])


def test_rank_is_integer_ceiling(orc):
    for n, E, k in [(4096, 64, 6), (131072, 256, 6), (262144, 256, 8), (524288, 256, 6),
                    (1, 256, 6), (7, 3, 2), (10, 4, 1), (12, 4, 1)]:
        R = orc.rank(n, E, k)
        assert R == -((-k * n) // E)
        assert 1 <= R <= n
    assert orc.rank(4096, 64, 6) == 384
    assert orc.rank(131072, 256, 6) == 3072
    assert orc.rank(262144, 256, 8) == 8192
    assert orc.rank(524288, 256, 6) == 12288
