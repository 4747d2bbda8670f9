"""GPU parity of the EQB path against the CPU oracle (bit-exact).

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph (hi-byte histogram, select, lo-byte histogram, exact quantile,
partition invariance); "[Dev] Add global-batch quantile balancing",
"Quantile estimator" and "Implementation" (alpha, margins, centering, pooled
histograms, in-place reset with stable addresses, replay counted once).
"""
import numpy as np
import pytest
import torch

from exact_distributed_quantiles_gb300 import inputs
from qb_testlib import assert_route_matches, gpu_route, host_logits, np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qb():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb as _qb
    return _qb


def _logits(N, E, seed, dtype=torch.float32, std=1.0, off_std=0.5):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    off = torch.randn(E, generator=g, device="cuda") * off_std
    x = torch.randn(N, E, generator=g, device="cuda") * std + off
    b = (torch.rand(E, generator=g, device="cuda") * 2 - 1) * 0.1
    return x.to(dtype).contiguous(), b


# powers of two, and multiples of 32 that run padded to the next one
ALL_E = [32, 64, 96, 128, 160, 256, 384, 480, 512, 640, 1024]


@pytest.mark.parametrize("E", ALL_E)
@pytest.mark.parametrize("k", [1, 6, 8, 15])
def test_route_small_shapes_fp32(qb, orc, E, k):
    if k >= E:
        pytest.skip("k must be below E")
    N = 32 * 7 + 13  # several tiles and a ragged tail
    x, b = _logits(N, E, seed=E * 100 + k)
    res = gpu_route(qb, x, b, k)
    ref = assert_route_matches(orc, res, host_logits(x), b.cpu().numpy(), k)
    assert np.array_equal(res["hist_hi"], orc.hist_hi(orc.keys(ref["margins"])))


@pytest.mark.parametrize("E,k", [(64, 6), (96, 6), (256, 8), (384, 8), (512, 6), (1024, 6)])
@pytest.mark.parametrize("N", [1, 31, 32, 33, 1000])
def test_route_bf16_and_ragged(qb, orc, E, k, N):
    x, b = _logits(N, E, seed=N + E, dtype=torch.bfloat16, std=1.5, off_std=0.3)
    res = gpu_route(qb, x, b, k)
    ref = assert_route_matches(orc, res, host_logits(x), b.cpu().numpy(), k)
    assert np.array_equal(res["hist_hi"], orc.hist_hi(orc.keys(ref["margins"])))


def test_route_ties(qb, orc):
    # Exact ties in s + b at and around alpha: equal bias entries, duplicated
    # logit columns, and whole rows of identical values.
    E, k, N = 64, 6, 300
    x, b = _logits(N, E, seed=3)
    b[1::2] = b[0::2]
    x[:, 1::2] = x[:, 0::2]
    x[::7, :] = x[::7, :1]
    b = b.contiguous()
    x = x.contiguous()
    res = gpu_route(qb, x, b, k)
    assert_route_matches(orc, res, host_logits(x), b.cpu().numpy(), k)


def test_route_extreme_logits(qb, orc):
    # |x| beyond the fast exponent range, subnormal scores, margins that round
    # to bf16 -0 (folded to the +0 key), saturated scores of exactly 1.
    E, k, N = 64, 6, 96
    x, b = _logits(N, E, seed=5)
    # scores a few subnormal ulps apart: margins round to bf16 -0
    x[0:32] = -88.0 + (torch.rand(32, E, device="cuda") - 0.5) * 1e-5
    x[32:48] = 90.0 + torch.rand(16, E, device="cuda") * 20.0
    x[48:64, ::3] = -120.0
    x[64:80] = -100.0 + torch.rand(16, E, device="cuda") * 20.0
    b[:] = 0.0
    res = gpu_route(qb, x.contiguous(), b, k)
    ref = assert_route_matches(orc, res, host_logits(x), b.cpu().numpy(), k)
    bits = orc.bf16_rne(ref["margins"])
    assert np.any(bits == 0x8000), "test should produce bf16 -0 margins"


def test_route_margins_outside_shared_window(qb, orc):
    # Large biases push |r| >= 2, whose hi bytes are counted outside the
    # shared-memory window (direct global atomics).
    E, k, N = 256, 6, 500
    x, b = _logits(N, E, seed=9)
    b = (torch.linspace(-4.0, 4.0, E, device="cuda")).contiguous()
    res = gpu_route(qb, x, b, k)
    ref = assert_route_matches(orc, res, host_logits(x), b.cpu().numpy(), k)
    h = orc.hist_hi(orc.keys(ref["margins"]))
    assert np.array_equal(res["hist_hi"], h)
    inside = np.zeros(256, bool)
    inside[0x40:0x50] = True
    inside[0xB0:0xC0] = True
    assert h[:, ~inside].sum() > 0


def _eqb_gpu(qb, mbs, bias, k, chained=False):
    # chained: every microbatch call after the first is qb_route_hist_hi_next
    E = bias.shape[0]
    st = qb.EQBState(E, bias.device)
    n_pool = sum(m.shape[0] for m in mbs)
    keys = torch.empty(n_pool, E, dtype=torch.int16, device=bias.device)
    b_out = torch.empty_like(bias)
    row = 0
    for i, m in enumerate(mbs):
        route = qb.qb_route_hist_hi_next if chained and i > 0 else qb.qb_route_hist_hi
        route(m, bias, k, st.hist_hi, keys_out=keys[row:row + m.shape[0]])
        row += m.shape[0]
    r = qb.rank(n_pool, E, k)
    qb.qb_select_hi(st.hist_hi, r, st.sel, st.r_lo)
    qb.qb_keys_hist_lo(keys, st.sel, st.hist_lo)
    h_hi = st.hist_hi.clone()
    h_lo = st.hist_lo.clone()
    qb.qb_finalize(st.hist_hi, st.hist_lo, st.sel, st.r_lo, b_out, qkey_out=st.qkey, reset=True)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    return dict(hist_hi=h_hi.cpu().numpy(), hist_lo=h_lo.cpu().numpy(), sel=st.sel.cpu().numpy(),
                r_lo=st.r_lo.cpu().numpy(), qkey=np_u16(st.qkey), bias_out=b_out.cpu().numpy(),
                keys=keys, state=st)


def _check_eqb(res, ref):
    for key in ("hist_hi", "hist_lo", "sel", "r_lo", "qkey"):
        assert np.array_equal(res[key], ref[key]), key
    assert np.array_equal(res["bias_out"].view(np.uint32), ref["bias_out"].view(np.uint32))


def test_eqb_tiny_workload(qb, orc):
    w = inputs.WORKLOADS["eqb_tiny"]
    bias, mbs = inputs.router_layer(w, inputs.seed_for("eqb_tiny"), device="cuda")
    res = _eqb_gpu(qb, mbs, bias, w.k)
    ref = orc.eqb_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k)
    _check_eqb(res, ref)
    assert res["hist_hi"].sum(axis=1).tolist() == [w.n_pool] * w.E


def test_eqb_pooled_workload_and_partition_invariance(qb, orc):
    w = inputs.WORKLOADS["eqb_pooled"]
    bias, mbs = inputs.router_layer(w, inputs.seed_for("eqb_pooled"), device="cuda")
    res = _eqb_gpu(qb, mbs, bias, w.k)
    ref = orc.eqb_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k)
    _check_eqb(res, ref)
    allx = torch.cat(mbs)
    for n_m, n_t, chained in ((2, 65536, False), (32, 4096, False), (1, 131072, False),
                              (8, 16384, True), (32, 4096, True), (128, 1024, True)):
        parts = [allx[i * n_t:(i + 1) * n_t] for i in range(n_m)]
        other = _eqb_gpu(qb, parts, bias, w.k, chained=chained)
        for key in ("hist_hi", "hist_lo", "sel", "r_lo", "qkey", "bias_out"):
            assert np.array_equal(res[key], other[key]), (n_m, chained, key)
        assert torch.equal(res["keys"], other["keys"]), (n_m, chained)
    # rank-local (per-microbatch) histograms differ before pooling
    h0 = gpu_route(qb, mbs[0], bias, w.k)["hist_hi"]
    h1 = gpu_route(qb, mbs[1], bias, w.k)["hist_hi"]
    assert not np.array_equal(h0, h1)


def test_lo_pass_recomputed_from_logits_equals_keys_pass(qb, orc):
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], n_micro=2, n_tokens=3000)
    bias, mbs = inputs.router_layer(w, 77, device="cuda")
    res = _eqb_gpu(qb, mbs, bias, w.k)
    sel = torch.from_numpy(res["sel"]).cuda()
    h = torch.zeros(w.E, 256, dtype=torch.int32, device="cuda")
    for m in mbs:
        qb.qb_route_hist_lo(m, bias, w.k, sel, h)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), res["hist_lo"])


def test_reset_in_place_and_replay_counted_once(qb, orc):
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], n_micro=2, n_tokens=2048)
    bias, mbs = inputs.router_layer(w, 78, device="cuda")
    res = _eqb_gpu(qb, mbs, bias, w.k)
    st = res["state"]
    ptrs = (st.hist_hi.data_ptr(), st.hist_lo.data_ptr())
    assert int(st.hist_hi.abs().sum()) == 0 and int(st.hist_lo.abs().sum()) == 0
    assert (st.hist_hi.data_ptr(), st.hist_lo.data_ptr()) == ptrs
    # a microbatch replayed after a reset is counted once
    qb.qb_route_hist_hi(mbs[0], bias, w.k, st.hist_hi)
    qb.qb_zero_i32(st.hist_hi)
    qb.qb_route_hist_hi(mbs[0], bias, w.k, st.hist_hi)
    torch.cuda.synchronize()
    once = gpu_route(qb, mbs[0], bias, w.k)["hist_hi"]
    assert np.array_equal(st.hist_hi.cpu().numpy(), once)


@pytest.mark.parametrize("E,dtype", [(256, torch.float32), (256, torch.bfloat16),
                                     (64, torch.float32)])
def test_chained_microbatches_across_steps(qb, orc, E, dtype):
    # Two global batches back to back on one stream through the binding's
    # helper, whose microbatch calls after the first are qb_route_hist_hi_next.
    # The second batch routes with the bias that the first batch's finalize
    # wrote, on the histogram it reset: a chained call that ran ahead of the
    # finalize would change the second bias.
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=E, n_micro=6, n_tokens=5000,
                      logits_dtype=dtype)
    bias, mbs1 = inputs.router_layer(w, 91, device="cuda")
    _, mbs2 = inputs.router_layer(w, 92, device="cuda")
    st = qb.EQBState(E, bias.device)
    keys = torch.empty(w.n_pool, E, dtype=torch.int16, device="cuda")
    b1, b2 = torch.empty_like(bias), torch.empty_like(bias)
    qb.eqb_global_batch(mbs1, bias, w.k, state=st, keys=keys, bias_out=b1)
    qb.eqb_global_batch(mbs2, b1, w.k, state=st, keys=keys, bias_out=b2)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    ref1 = orc.eqb_global_batch([host_logits(m) for m in mbs1], bias.cpu().numpy(), w.k)
    ref2 = orc.eqb_global_batch([host_logits(m) for m in mbs2], ref1["bias_out"], w.k)
    assert np.array_equal(b1.cpu().numpy().view(np.uint32), ref1["bias_out"].view(np.uint32))
    assert np.array_equal(b2.cpu().numpy().view(np.uint32), ref2["bias_out"].view(np.uint32))
    assert np.array_equal(np_u16(keys), np.concatenate(ref2["keys"]))


@pytest.mark.parametrize("layer", [0, 23, 47])
def test_full_step_layer_at_bench_size(qb, orc, layer):
    # Layers 0, 23 and 47 of the full-step workload (their own seeds), each
    # routed in both launch shapes: the 16 microbatch calls of 32768 tokens
    # that the benchmark times, and one call over the whole layer.  Compared
    # with the oracle over every token.
    w = inputs.WORKLOADS["full_step"]
    out = torch.empty(w.n_pool, w.E, dtype=torch.float32, device="cuda")
    bias, mbs = inputs.router_layer(w, inputs.seed_for("full_step", layer), device="cuda",
                                    out=out)
    ref = orc.eqb_global_batch([out.cpu().numpy()], bias.cpu().numpy(), w.k)
    for parts, chained in ((mbs, False), (mbs, True), ([out], False)):
        res = _eqb_gpu(qb, parts, bias, w.k, chained=chained)
        _check_eqb(res, ref)
        assert np.array_equal(np_u16(res["keys"]), np.concatenate(ref["keys"]))


@pytest.mark.parametrize("E,k", [(32, 1), (64, 6), (96, 6), (128, 8), (160, 15), (256, 6),
                                 (384, 8), (480, 6), (512, 15), (640, 6), (1024, 8)])
def test_eqb_all_expert_counts(qb, orc, E, k):
    # the whole EQB chain (hi pass, select, lo pass from keys, finalize) for
    # every supported expert count, several tiles and a ragged tail
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=E, k=k, n_micro=3, n_tokens=16 * 37 + 5)
    bias, mbs = inputs.router_layer(w, 300 + E, device="cuda")
    res = _eqb_gpu(qb, mbs, bias, w.k)
    ref = orc.eqb_global_batch([host_logits(m) for m in mbs], bias.cpu().numpy(), w.k)
    _check_eqb(res, ref)


def _lo_keys(N, E, seed):
    # keys concentrated on a few hi bytes (so that many fall in the selected
    # bin), every lo byte, and some keys in bins 0x00 and 0xFF
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    hi = torch.randint(0, 4, (N, E), generator=g, device="cuda") + 0x80
    hi[torch.rand(N, E, generator=g, device="cuda") < 0.05] = 0xFF
    hi[torch.rand(N, E, generator=g, device="cuda") < 0.05] = 0x00
    lo = torch.randint(0, 256, (N, E), generator=g, device="cuda")
    keys = (hi * 256 + lo).to(torch.int32).to(torch.int16)
    sel = torch.randint(0x80, 0x84, (E,), generator=g, device="cuda").to(torch.int32)
    sel[::7] = -1                 # no selected bin
    sel[3::11] = 0xFF
    sel[5::13] = 0x00
    return keys, sel


@pytest.mark.parametrize("E", ALL_E)
@pytest.mark.parametrize("N", [1, 31, 4097])
def test_keys_hist_lo_equals_definition(qb, orc, E, N):
    # The lo pass from stored keys equals the oracle's direct count on keys
    # spread over bins 0x00, 0x80-0x83 and 0xFF, with sel = -1 (no selected
    # bin) counting nothing and sel = 0x00 / 0xFF counting the edge bins.
    keys, sel = _lo_keys(N, E, seed=E * 7 + N)
    want = orc.hist_lo(np_u16(keys), sel.cpu().numpy())
    h = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    qb.qb_keys_hist_lo(keys, sel, h)
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), want)


def _keys_of(values):
    # order-preserving key of each bf16 number given as fp32 (+0 for -0)
    v = np.asarray(values, np.float32).copy()
    v[v == 0] = 0.0
    b = (v.view(np.uint32) >> 16).astype(np.uint32)
    return np.where(b & 0x8000, b ^ 0xFFFF, b ^ 0x8000).astype(np.uint16)


@pytest.mark.parametrize("E", ALL_E)
@pytest.mark.parametrize("spread", ["narrow", "wide", "no_bin"])
def test_finalize_on_built_histograms(qb, orc, E, spread):
    # qb_finalize against the plain definition on hand-built histograms: the
    # selected key of each expert is known, extra counts sit below and above
    # it in its bin so that the rank lands mid-row, and the quantiles span a
    # narrow exponent range (the tree sum is exact) or about 2^-60 .. 2^60
    # (the serial ascending sum decides), or one expert has no selected bin
    # (every output NaN, as the mean is undefined).  Keys at lo bytes 0x00
    # and 0xFF are included.
    rng = np.random.default_rng(E * 3 + len(spread))
    if spread == "wide":
        mag = 2.0 ** rng.integers(-60, 61, E)
    else:
        mag = 2.0 ** rng.integers(-3, 3, E)
    vals = (rng.uniform(1, 2, E) * mag * rng.choice([-1.0, 1.0], E)).astype(np.float32)
    vals = (vals.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16 numbers
    keys = _keys_of(vals)
    keys[0] = (keys[0] & 0xFF00) | 0x00
    keys[1] = (keys[1] & 0xFF00) | 0xFF
    sel = (keys >> 8).astype(np.int32)
    lo = (keys & 0xFF).astype(np.int32)
    hist_lo = np.zeros((E, 256), np.int32)
    r_lo = np.zeros(E, np.int32)
    for j in range(E):
        below = int(rng.integers(0, 5)) if lo[j] > 0 else 0
        if below:
            hist_lo[j, rng.integers(0, lo[j], below)] += 1
        at = int(rng.integers(1, 4))
        hist_lo[j, lo[j]] += at
        if lo[j] < 255:
            hist_lo[j, rng.integers(lo[j] + 1, 256, 3)] += 1
        r_lo[j] = hist_lo[j, :lo[j]].sum() + int(rng.integers(1, at + 1))
    if spread == "no_bin":
        sel[E // 2] = -1
    hist_hi = rng.integers(0, 9, (E, 256)).astype(np.int32)
    d = {n: torch.from_numpy(a).cuda() for n, a in
         (("hh", hist_hi), ("hl", hist_lo), ("sel", sel), ("rlo", r_lo))}
    b_out = torch.empty(E, dtype=torch.float32, device="cuda")
    qk = torch.empty(E, dtype=torch.int16, device="cuda")
    qb.qb_finalize(d["hh"], d["hl"], d["sel"], d["rlo"], b_out, qkey_out=qk, reset=True)
    torch.cuda.synchronize()
    got = b_out.cpu().numpy()
    assert int(d["hh"].abs().sum()) == 0 and int(d["hl"].abs().sum()) == 0
    if spread == "no_bin":
        assert np.isnan(got).all()
        assert np_u16(qk)[E // 2] == 0
        return
    assert np.array_equal(np_u16(qk), keys)
    q = orc.key_decode_array(keys).astype(np.float64)
    want = orc.center(q)
    assert np.array_equal(got.view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("E", ALL_E)
@pytest.mark.parametrize("k", [1, 6, 15])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_lo_pass_recomputed_all_shapes(qb, orc, E, k, dtype):
    # The lo pass that recomputes the keys from the logits (qb_route_hist_lo)
    # equals the oracle's direct count on its own keys, for every expert count
    # (E = 512 reads the selected bins of two 256-expert halves), fp32 and
    # bf16 logits and a ragged token count.  sel comes from the oracle's
    # select, so both sides count the same bins.
    if k >= E:
        pytest.skip("k must be below E")
    N = 32 * 9 + 21
    x, b = _logits(N, E, seed=E * 31 + k + (dtype == torch.bfloat16),
                   dtype=dtype, std=1.5 if dtype == torch.bfloat16 else 1.0)
    ref = orc.route(host_logits(x), b.cpu().numpy(), k, want=("margins",))
    keys = orc.keys(ref["margins"])
    sel, _ = orc.select_hi(orc.hist_hi(keys), orc.rank(N, E, k))
    sel = np.asarray(sel, np.int32).copy()
    sel[::5] = -1  # experts without a selected bin count nothing
    want = orc.hist_lo(keys, sel)
    h = torch.zeros(E, 256, dtype=torch.int32, device="cuda")
    qb.qb_route_hist_lo(x, b, k, torch.from_numpy(sel).cuda(), h)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    assert np.array_equal(h.cpu().numpy(), want)
    assert int(h.sum()) > 0
