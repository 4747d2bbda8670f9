"""Pins for BF16 rounding and the order-preserving key (CPU only).

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph: radix selection over the two bytes of BF16 margins works because
the bit patterns can be made to follow value order.  Raw patterns only do so
for non-negative values; the key used here flips the sign bit of positives and
every bit of negatives, after folding -0 onto +0.
"""
import numpy as np
import pytest
import torch


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _boundary_patterns():
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xFFFE, 0xFFFF], np.uint32)
    u = (hi[:, None] | lows[None, :]).ravel()
    x = u.view(np.float32)
    return x[~np.isnan(x)]


def test_bf16_rne_matches_library_rounding_on_every_boundary(orc):
    # Every binary32 value adjacent to a bf16 rounding boundary (exact ties,
    # one below, one above), for every sign/exponent/high-mantissa pattern.
    x = _boundary_patterns()
    assert np.array_equal(orc.bf16_rne(x), _torch_bf16_bits(x))


def test_bf16_rne_matches_library_rounding_random(orc):
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    assert np.array_equal(orc.bf16_rne(x), _torch_bf16_bits(x))


def test_bf16_rne_hand_cases(orc):
    cases = [
        (1.0, 0x3F80),
        (-1.0, 0xBF80),
        # 1 + 2^-8 is an exact tie between 1 and 1 + 2^-7: ties go to even (1.0)
        (1.0 + 2.0 ** -8, 0x3F80),
        # 1 + 3*2^-8 ties between 1+2^-7 (odd mantissa) and 1+2^-6 (even)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),
        (0.0, 0x0000),
        (-0.0, 0x8000),
    ]
    for v, bits in cases:
        got = int(orc.bf16_rne(np.float32([v]))[0])
        assert got == _torch_bf16_bits(np.float32([v]))[0]
        assert got == bits, (v, hex(got))
    # Largest finite float rounds up to infinity (bf16 max is 0x7F7F).
    assert orc.bf16_rne(np.float32([np.finfo(np.float32).max]))[0] == 0x7F80
    # Tiny negative subnormal below half the least bf16 subnormal rounds to -0.
    assert orc.bf16_rne(np.array([0x80000001], np.uint32).view(np.float32))[0] == 0x8000


def test_key_orders_every_bf16_value():
    import oracle as orc_mod
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    ok = ~np.isnan(vals)
    vals = vals[ok]
    keys = orc_mod.keys(vals).astype(np.int64)
    order = np.argsort(vals, kind="stable")
    v_sorted, k_sorted = vals[order], keys[order]
    # value order <=> key order, with equal values (only +0 / -0) sharing a key
    dv = np.diff(v_sorted.astype(np.float64))
    dk = np.diff(k_sorted)
    assert np.all((dv > 0) == (dk > 0))
    assert np.all((dv == 0) == (dk == 0))
    # The map is a bijection of the 65536 patterns apart from the -0 fold.
    assert len(np.unique(keys)) == len(keys) - 1


def test_key_hand_values(orc):
    assert orc.keys(np.float32([0.0]))[0] == 0x8000
    assert orc.keys(np.float32([-0.0]))[0] == 0x8000  # -0 folds to +0
    assert orc.keys(np.array([0x80000001], np.uint32).view(np.float32))[0] == 0x8000
    assert orc.keys(np.float32([1.0]))[0] == 0x3F80 ^ 0x8000
    assert orc.keys(np.float32([-1.0]))[0] == 0xBF80 ^ 0xFFFF
    assert orc.keys(np.float32([-np.inf]))[0] == 0x007F
    assert orc.keys(np.float32([np.inf]))[0] == 0xFF80


def test_key_decode_inverts_key(orc):
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[~np.isnan(vals)]
    k = orc.keys(vals)
    dec = orc.key_decode_array(k)
    same = (dec == vals) | ((dec == 0) & (vals == 0))
    assert np.all(same)
    for key in (0x8000, 0xBF80, 0x407F, 0x1234, 0xC321):
        assert orc.key_decode(key) == orc.key_decode_array(np.uint16([key]))[0]
