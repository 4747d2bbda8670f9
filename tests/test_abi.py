"""The C-ABI library loads and exports every symbol include/qb.h declares, and
its host-side argument checks return the documented status codes (CPU only:
these calls are rejected before any CUDA work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qb.h")


@pytest.fixture(scope="module")
def lib():
    from exact_distributed_quantiles_gb300 import build
    build.build()
    from exact_distributed_quantiles_gb300 import qb
    return qb


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("qb_route_hist_hi", "qb_select_hi", "qb_route_hist_lo", "qb_keys_hist_lo",
              "qb_finalize", "k3_route_hist", "k3_finalize", "lei_inject"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in _declared():
        assert hasattr(so, n), n
    assert set(lib.EXPORTS) == set(_declared())


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert lib.status_string(st) and lib.status_string(st) != "unknown status"
    assert lib.version().startswith("libqb")


def test_rank(lib):
    assert lib.rank(524288, 256, 6) == 12288
    assert lib.rank(131072, 256, 6) == 3072
    assert lib.rank(4096, 64, 6) == 384
    assert lib.rank(7, 3, 2) == 5
    assert lib.lib.qb_rank(0, 256, 6) == lib.QB_EINVAL
    assert lib.lib.qb_rank(10, 4, 4) == lib.QB_EINVAL


def test_argument_errors_are_reported_before_launch(lib):
    L = lib.lib
    fake = ctypes.c_void_p(0x10000)   # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(0x10004)
    N0 = None
    for hi in (L.qb_route_hist_hi, L.qb_route_hist_hi_next):
        # null logits / bias / histogram
        assert hi(N0, 0, fake, 10, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, N0, 10, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, 10, 256, 6, N0, N0, N0, N0, N0) == lib.QB_EINVAL
        # misaligned logits or keys
        assert hi(odd, 0, fake, 10, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, 10, 256, 6, fake, odd, N0, N0, N0) == lib.QB_EINVAL
        # bad dtype, negative N, N beyond int32 counts
        assert hi(fake, 7, fake, 10, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, -1, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, 1 << 31, 256, 6, fake, N0, N0, N0, N0) == lib.QB_EOVERFLOW
        # unsupported E, bad k
        for E in (0, 16, 48, 1056, 2048):
            assert hi(fake, 0, fake, 10, E, 6, fake, N0, N0, N0, N0) == lib.QB_EUNSUPPORTED
        assert hi(fake, 0, fake, 10, 256, 0, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, 10, 32, 32, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert hi(fake, 0, fake, 10, 256, 16, fake, N0, N0, N0, N0) == lib.QB_EUNSUPPORTED
        # empty input is a no-op
        assert hi(fake, 0, fake, 0, 256, 6, fake, N0, N0, N0, N0) == lib.QB_OK
    # select: rank out of range
    assert L.qb_select_hi(fake, 256, 0, fake, fake, N0) == lib.QB_EINVAL
    assert L.qb_select_hi(fake, 256, 1 << 31, fake, fake, N0) == lib.QB_EOVERFLOW
    assert L.qb_select_hi(N0, 256, 5, fake, fake, N0) == lib.QB_EINVAL
    # lo pass
    assert L.qb_keys_hist_lo(odd, 10, 256, fake, fake, N0) == lib.QB_EINVAL
    assert L.qb_keys_hist_lo(fake, 10, 512 + 1, fake, fake, N0) == lib.QB_EUNSUPPORTED
    assert L.qb_keys_hist_lo(fake, 0, 256, fake, fake, N0) == lib.QB_OK
    assert L.qb_route_hist_lo(fake, 0, fake, 10, 256, 6, N0, fake, N0) == lib.QB_EINVAL
    # finalize
    assert L.qb_finalize(fake, fake, fake, fake, 256, N0, N0, 1, N0) == lib.QB_EINVAL
    assert L.qb_finalize(N0, fake, fake, fake, 256, fake, N0, 1, N0) == lib.QB_EINVAL
    # K3 (plain and chained entries)
    for k3 in (L.k3_route_hist, L.k3_route_hist_next):
        assert k3(fake, 1, fake, 10, 256, 8, fake, 0, fake, fake, N0) == lib.QB_EINVAL
        assert k3(fake, 1, fake, 10, 256, 8, N0, 1000, fake, fake, N0) == lib.QB_EINVAL
        assert k3(fake, 1, fake, 10, 256, 8, fake, 1000, fake, N0, N0) == lib.QB_EINVAL
        assert k3(fake, 1, fake, 10, 256, 8, fake, 1000, fake,
                  ctypes.c_void_p(65537), N0) == lib.QB_EINVAL  # alpha_out misaligned
        assert k3(fake, 1, fake, 0, 256, 8, fake, 1000, fake, fake, N0) == lib.QB_OK
    assert L.k3_finalize(fake, 256, 1000, 0, fake, fake, 1, N0) == lib.QB_EINVAL
    assert L.k3_finalize(fake, 256, 70000, 5, fake, fake, 1, N0) == lib.QB_EINVAL
    # LEI
    assert L.lei_inject(odd, fake, 10, 256, 6, 8e-5, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_inject(fake, fake, 10, 256, 6, 8e-5, 0, N0, N0) == lib.QB_EINVAL
    assert L.lei_inject(fake, fake, 10, 256, 0, 8e-5, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_inject(fake, fake, 0, 256, 6, 8e-5, 0, fake, N0) == lib.QB_OK
    assert L.lei_rho(fake, 10, 256, 6, 8e-5, 0, N0, N0) == lib.QB_EINVAL
    assert L.lei_rho(fake, 10, 256, 6, 8e-5, 0, odd, N0) == lib.QB_EINVAL
    assert L.lei_rho(fake, 10, 100, 6, 8e-5, 0, fake, N0) == lib.QB_EUNSUPPORTED
    assert L.lei_rho(fake, 10, 256, 0, 8e-5, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_rho(fake, 0, 256, 6, 8e-5, 0, fake, N0) == lib.QB_OK
    assert L.lei_apply(odd, 10, 256, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_apply(fake, 10, 256, 0, odd, N0) == lib.QB_EINVAL
    assert L.lei_apply(fake, -1, 256, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_apply(fake, 10, 100, 0, fake, N0) == lib.QB_EUNSUPPORTED
    assert L.lei_apply(fake, 0, 256, 0, fake, N0) == lib.QB_OK
    assert L.lei_apply_overlap(odd, 10, 256, 0, fake, N0) == lib.QB_EINVAL
    assert L.lei_apply_overlap(fake, 10, 256, 0, N0, N0) == lib.QB_EINVAL
    assert L.lei_apply_overlap(fake, 10, 256, -1, fake, N0) == lib.QB_EINVAL
    assert L.lei_apply_overlap(fake, 10, 48, 0, fake, N0) == lib.QB_EUNSUPPORTED
    assert L.lei_apply_overlap(fake, 0, 256, 0, fake, N0) == lib.QB_OK
    # router GEMM with the hi pass (plain and chained entries)
    for g in (L.qb_router_gemm_hist_hi, L.qb_router_gemm_hist_hi_next):
        assert g(N0, fake, 10, 2048, 256, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert g(odd, fake, 10, 2048, 256, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert g(fake, fake, 10, 2048, 256, 6, fake, N0, N0, N0, N0, N0, N0) == lib.QB_EINVAL
        assert g(fake, fake, 10, 2000, 256, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EUNSUPPORTED
        assert g(fake, fake, 10, 2048, 288, 6, fake, fake, fake, N0, N0, N0, N0) == lib.QB_EUNSUPPORTED
        assert g(fake, fake, 10, 2048, 96, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EUNSUPPORTED
        assert g(fake, fake, 10, 2048, 256, 0, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert g(fake, fake, -1, 2048, 256, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_EINVAL
        assert g(fake, fake, 0, 2048, 256, 6, fake, N0, fake, N0, N0, N0, N0) == lib.QB_OK
    # rank average and MaxVio
    assert L.qb_rank_average(N0, 2, 256, fake, N0) == lib.QB_EINVAL
    assert L.qb_rank_average(fake, 0, 256, fake, N0) == lib.QB_EINVAL
    assert L.qb_rank_average(fake, 2, 100, fake, N0) == lib.QB_EUNSUPPORTED
    assert L.qb_maxvio(odd, 10, 256, 6, 0, fake, fake, N0) == lib.QB_EINVAL
    assert L.qb_maxvio(fake, 0, 256, 6, 0, fake, fake, N0) == lib.QB_EINVAL
    assert L.qb_maxvio(fake, 10, 256, 6, 0, fake, N0, N0) == lib.QB_EINVAL
    assert L.qb_maxvio(fake, 10, 256, 256, 0, fake, fake, N0) == lib.QB_EINVAL


def test_binding_raises_with_status(lib):
    with pytest.raises(lib.QBError) as ei:
        lib.rank(0, 256, 6)
    assert ei.value.status == lib.QB_EINVAL
