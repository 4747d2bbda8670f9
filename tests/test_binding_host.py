"""Host logic of the binding's global-batch helper (CPU only, no kernel runs).

`qb.eqb_global_batch` issues the first microbatch of a global batch with
qb_route_hist_hi and every later one with qb_route_hist_hi_next (which may
start before the call before it ends: "[Dev] Add global-batch quantile
balancing", "Implementation", one histogram accumulated over every
microbatch).  A microbatch of zero tokens issues no work, so the call after
it must still be chained to the last call that did.  The routing and
counting calls are replaced by recorders here.
"""
import pytest
import torch


@pytest.fixture(scope="module")
def qb():
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _record(qb, monkeypatch):
    calls = []

    def route(name):
        def f(m, bias, k, hist, keys_out=None, stream=None):
            calls.append((name, int(m.shape[0]), int(keys_out.shape[0])))
        return f

    monkeypatch.setattr(qb, "qb_route_hist_hi", route("hi"))
    monkeypatch.setattr(qb, "qb_route_hist_hi_next", route("next"))
    for name in ("qb_select_hi", "qb_keys_hist_lo", "qb_finalize"):
        monkeypatch.setattr(qb, name, lambda *a, _n=name, **kw: calls.append((_n,)))
    return calls


@pytest.mark.parametrize("sizes,expect", [
    ([5, 7, 3], ["hi", "next", "next"]),
    ([0, 4, 0, 6], ["hi", "next"]),
    ([9], ["hi"]),
])
def test_global_batch_chains_the_later_microbatches(qb, monkeypatch, sizes, expect):
    calls = _record(qb, monkeypatch)
    E = 32
    bias = torch.zeros(E)
    mbs = [torch.zeros(n, E) for n in sizes]
    qb.eqb_global_batch(mbs, bias, 2, state=qb.EQBState(E, "cpu"))
    route_calls = [c for c in calls if c[0] in ("hi", "next")]
    assert [c[0] for c in route_calls] == expect
    # each microbatch's keys go to its own rows, in order
    assert [c[1] for c in route_calls] == [n for n in sizes if n]
    assert [c[2] for c in route_calls] == [n for n in sizes if n]
    assert [c[0] for c in calls[len(route_calls):]] == ["qb_select_hi", "qb_keys_hist_lo",
                                                       "qb_finalize"]
