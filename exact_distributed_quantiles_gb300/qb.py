"""Thin ctypes binding of ``libqb.so`` with the C entry points' names.

Argument marshalling only: tensors become device pointers, the stream defaults
to torch's current stream, and a non-zero status raises ``QBError``.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
fallback.  Importing this module raises if ``libqb.so`` has not been built
(``python -m exact_distributed_quantiles_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqb.so")

QB_OK, QB_EINVAL, QB_EUNSUPPORTED, QB_ECUDA, QB_EOVERFLOW, QB_EDEVICE = 0, -1, -2, -3, -4, -5
QB_F32, QB_BF16 = 0, 1

EXPORTS = ("qb_status_string", "qb_version", "qb_rank", "qb_sigmoid", "qb_sigmoid_scalar",
           "qb_zero_i32",
           "qb_route_hist_hi", "qb_route_hist_hi_next", "qb_select_hi", "qb_keys_hist_lo",
           "qb_route_hist_lo",
           "qb_finalize", "k3_route_hist", "k3_route_hist_next", "k3_finalize", "lei_inject",
           "qb_device_status",
           "lei_inject_noalloc", "qb_router_gemm", "qb_router_gemm_hist_hi",
           "qb_router_gemm_hist_hi_next", "qb_rank_average",
           "qb_maxvio", "lei_rho", "lei_apply",
           "lei_apply_overlap", "qb_selftest_wait_timeout")


class QBError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed with status {status}: {status_string(status)}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqb.so not built at {LIB_PATH}; run "
                          "`python -m exact_distributed_quantiles_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sigs = {
        "qb_status_string": (ctypes.c_char_p, [I]),
        "qb_version": (ctypes.c_char_p, []),
        "qb_rank": (I64, [I64, I, I]),
        "qb_sigmoid": (I, [P, P, I64, P]),
        "qb_sigmoid_scalar": (I, [P, P, I64, P]),
        "qb_zero_i32": (I, [P, I64, P]),
        "qb_route_hist_hi": (I, [P, I, P, I64, I, I, P, P, P, P, P]),
        "qb_route_hist_hi_next": (I, [P, I, P, I64, I, I, P, P, P, P, P]),
        "qb_select_hi": (I, [P, I, I64, P, P, P]),
        "qb_keys_hist_lo": (I, [P, I64, I, P, P, P]),
        "qb_route_hist_lo": (I, [P, I, P, I64, I, I, P, P, P]),
        "qb_finalize": (I, [P, P, P, P, I, P, P, I, P]),
        "k3_route_hist": (I, [P, I, P, I64, I, I, P, I, P, P, P]),
        "k3_route_hist_next": (I, [P, I, P, I64, I, I, P, I, P, P, P]),
        "k3_finalize": (I, [P, I, I, I64, P, P, I, P]),
        "lei_inject": (I, [P, P, I64, I, I, F, I64, P, P]),
        "qb_device_status": (I, [ctypes.POINTER(ctypes.c_int)]),
        "lei_inject_noalloc": (I, [P, P, I64, I, I, F, I64, P]),
        "qb_router_gemm": (I, [P, P, I64, I, I, P, P]),
        "qb_router_gemm_hist_hi": (I, [P, P, I64, I, I, I, P, P, P, P, P, P, P]),
        "qb_router_gemm_hist_hi_next": (I, [P, P, I64, I, I, I, P, P, P, P, P, P, P]),
        "qb_rank_average": (I, [P, I, I, P, P]),
        "qb_maxvio": (I, [P, I64, I, I, I64, P, P, P]),
        "lei_rho": (I, [P, I64, I, I, F, I64, P, P]),
        "lei_apply": (I, [P, I64, I, I64, P, P]),
        "lei_apply_overlap": (I, [P, I64, I, I64, P, P]),
        "qb_selftest_wait_timeout": (I, [I64, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.qb_status_string(int(status)).decode()


def version() -> str:
    return lib.qb_version().decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn: str, st: int):
    if st != QB_OK:
        raise QBError(fn, st)


def _dtype(t) -> int:
    if t.dtype == torch.float32:
        return QB_F32
    if t.dtype == torch.bfloat16:
        return QB_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def rank(n_pool: int, E: int, k: int) -> int:
    r = int(lib.qb_rank(int(n_pool), int(E), int(k)))
    if r < 0:
        raise QBError("qb_rank", r)
    return r


def qb_sigmoid(x, s, stream=None):
    _check("qb_sigmoid", lib.qb_sigmoid(_ptr(x), _ptr(s), x.numel(), _stream(stream)))


def qb_sigmoid_scalar(x, s, stream=None):
    _check("qb_sigmoid_scalar", lib.qb_sigmoid_scalar(_ptr(x), _ptr(s), x.numel(), _stream(stream)))


def qb_zero_i32(t, stream=None):
    _check("qb_zero_i32", lib.qb_zero_i32(_ptr(t), t.numel(), _stream(stream)))


def qb_route_hist_hi(logits, bias, k, hist_hi, keys_out=None, topk_out=None, alpha_out=None,
                     stream=None):
    N, E = logits.shape
    _check("qb_route_hist_hi",
           lib.qb_route_hist_hi(_ptr(logits), _dtype(logits), _ptr(bias), N, E, int(k),
                                _ptr(hist_hi), _ptr(keys_out), _ptr(topk_out), _ptr(alpha_out),
                                _stream(stream)))


def qb_route_hist_hi_next(logits, bias, k, hist_hi, keys_out=None, topk_out=None,
                          alpha_out=None, stream=None):
    N, E = logits.shape
    _check("qb_route_hist_hi_next",
           lib.qb_route_hist_hi_next(_ptr(logits), _dtype(logits), _ptr(bias), N, E, int(k),
                                     _ptr(hist_hi), _ptr(keys_out), _ptr(topk_out),
                                     _ptr(alpha_out), _stream(stream)))


def qb_select_hi(hist_hi, r, sel, r_lo, stream=None):
    E = hist_hi.shape[0]
    _check("qb_select_hi", lib.qb_select_hi(_ptr(hist_hi), E, int(r), _ptr(sel), _ptr(r_lo),
                                            _stream(stream)))


def qb_keys_hist_lo(keys, sel, hist_lo, stream=None):
    N, E = keys.shape
    _check("qb_keys_hist_lo", lib.qb_keys_hist_lo(_ptr(keys), N, E, _ptr(sel), _ptr(hist_lo),
                                                  _stream(stream)))


def qb_route_hist_lo(logits, bias, k, sel, hist_lo, stream=None):
    N, E = logits.shape
    _check("qb_route_hist_lo",
           lib.qb_route_hist_lo(_ptr(logits), _dtype(logits), _ptr(bias), N, E, int(k), _ptr(sel),
                                _ptr(hist_lo), _stream(stream)))


def qb_finalize(hist_hi, hist_lo, sel, r_lo, bias_out, qkey_out=None, reset=True, stream=None):
    E = hist_lo.shape[0]
    _check("qb_finalize",
           lib.qb_finalize(_ptr(hist_hi), _ptr(hist_lo), _ptr(sel), _ptr(r_lo), E, _ptr(bias_out),
                           _ptr(qkey_out), 1 if reset else 0, _stream(stream)))


def k3_route_hist(logits, bias, k, bounds, hist, alpha_out, stream=None):
    N, E = logits.shape
    nbins = hist.shape[1]
    _check("k3_route_hist",
           lib.k3_route_hist(_ptr(logits), _dtype(logits), _ptr(bias), N, E, int(k), _ptr(bounds),
                             nbins, _ptr(hist), _ptr(alpha_out), _stream(stream)))


def k3_route_hist_next(logits, bias, k, bounds, hist, alpha_out, stream=None):
    N, E = logits.shape
    nbins = hist.shape[1]
    _check("k3_route_hist_next",
           lib.k3_route_hist_next(_ptr(logits), _dtype(logits), _ptr(bias), N, E, int(k),
                                  _ptr(bounds), nbins, _ptr(hist), _ptr(alpha_out),
                                  _stream(stream)))


def k3_finalize(hist, r, bounds, bias_out, reset=True, stream=None):
    E, nbins = hist.shape
    _check("k3_finalize", lib.k3_finalize(_ptr(hist), E, nbins, int(r), _ptr(bounds),
                                          _ptr(bias_out), 1 if reset else 0, _stream(stream)))


def lei_inject(grad, topk_idx, eta, workspace, batch_tokens=0, stream=None):
    N, E = grad.shape
    k = topk_idx.shape[1]
    _check("lei_inject",
           lib.lei_inject(_ptr(grad), _ptr(topk_idx), N, E, int(k), float(eta), int(batch_tokens),
                          _ptr(workspace), _stream(stream)))


def lei_rho(topk_idx, E, eta, workspace, batch_tokens=0, stream=None):
    """First half of lei_inject: eta*rho per local batch into workspace."""
    N, k = topk_idx.shape
    _check("lei_rho", lib.lei_rho(_ptr(topk_idx), N, int(E), int(k), float(eta),
                                  int(batch_tokens), _ptr(workspace), _stream(stream)))


def lei_apply(grad, workspace, batch_tokens=0, stream=None):
    """Second half of lei_inject: grad += workspace[batch(row)]."""
    N, E = grad.shape
    _check("lei_apply", lib.lei_apply(_ptr(grad), N, E, int(batch_tokens), _ptr(workspace),
                                      _stream(stream)))


def lei_apply_overlap(grad, workspace, batch_tokens=0, stream=None):
    """lei_apply launched to run beside the kernel enqueued just before it
    on the stream (it must not touch grad or write workspace)."""
    N, E = grad.shape
    _check("lei_apply_overlap",
           lib.lei_apply_overlap(_ptr(grad), N, E, int(batch_tokens), _ptr(workspace),
                                 _stream(stream)))


def lei_inject_noalloc(grad, topk_idx, eta, batch_tokens=0, stream=None):
    """lei_inject with the library's own fixed scratch instead of a caller
    workspace (for callers that cannot allocate device memory)."""
    N, E = grad.shape
    k = topk_idx.shape[1]
    _check("lei_inject_noalloc",
           lib.lei_inject_noalloc(_ptr(grad), _ptr(topk_idx), N, E, int(k), float(eta),
                                  int(batch_tokens), _stream(stream)))


def qb_router_gemm(hidden, w_t, logits_out, stream=None):
    M, H = hidden.shape
    E = w_t.shape[0]
    _check("qb_router_gemm", lib.qb_router_gemm(_ptr(hidden), _ptr(w_t), M, H, E, _ptr(logits_out),
                                                _stream(stream)))


def qb_router_gemm_hist_hi(hidden, w_t, bias, k, logits_out, hist_hi, keys_out=None,
                           topk_out=None, alpha_out=None, stream=None):
    M, H = hidden.shape
    E = w_t.shape[0]
    _check("qb_router_gemm_hist_hi",
           lib.qb_router_gemm_hist_hi(_ptr(hidden), _ptr(w_t), M, H, E, int(k), _ptr(bias),
                                      _ptr(logits_out), _ptr(hist_hi), _ptr(keys_out),
                                      _ptr(topk_out), _ptr(alpha_out), _stream(stream)))


def qb_router_gemm_hist_hi_next(hidden, w_t, bias, k, logits_out, hist_hi, keys_out=None,
                                topk_out=None, alpha_out=None, stream=None):
    M, H = hidden.shape
    E = w_t.shape[0]
    _check("qb_router_gemm_hist_hi_next",
           lib.qb_router_gemm_hist_hi_next(_ptr(hidden), _ptr(w_t), M, H, E, int(k), _ptr(bias),
                                           _ptr(logits_out), _ptr(hist_hi), _ptr(keys_out),
                                           _ptr(topk_out), _ptr(alpha_out), _stream(stream)))


def qb_rank_average(qkeys, bias_out, stream=None):
    """qkeys: int16/uint16 [P, E] selected keys of P ranks -> centred average bias."""
    P, E = qkeys.shape
    _check("qb_rank_average", lib.qb_rank_average(_ptr(qkeys), P, E, _ptr(bias_out),
                                                  _stream(stream)))


def qb_maxvio(topk, E, loads_out, maxvio_out, batch_tokens=0, stream=None):
    N, k = topk.shape
    _check("qb_maxvio", lib.qb_maxvio(_ptr(topk), N, int(E), k, int(batch_tokens),
                                      _ptr(loads_out), _ptr(maxvio_out), _stream(stream)))


def device_status() -> int:
    flags = ctypes.c_int(0)
    st = lib.qb_device_status(ctypes.byref(flags))
    if st == QB_ECUDA:
        raise QBError("qb_device_status", st)
    return int(flags.value)


# ---------------------------------------------------------------- convenience

class EQBState:
    """Device buffers of one router's EQB global batch (caller-owned memory).

    hist_hi / hist_lo: int32 [E,256]; sel / r_lo: int32 [E]."""

    def __init__(self, E: int, device="cuda"):
        self.E = E
        self.hist_hi = torch.zeros(E, 256, dtype=torch.int32, device=device)
        self.hist_lo = torch.zeros(E, 256, dtype=torch.int32, device=device)
        self.sel = torch.empty(E, dtype=torch.int32, device=device)
        self.r_lo = torch.empty(E, dtype=torch.int32, device=device)
        self.qkey = torch.empty(E, dtype=torch.int16, device=device)


def eqb_global_batch(microbatches, bias, k, state: EQBState | None = None, keys=None,
                     bias_out=None, reset=True, stream=None):
    """Hi pass per microbatch, select, lo pass over the stored keys, finalize.

    ``keys`` (uint16 as int16 [N_pool, E]) receives the keys of every
    microbatch in order; allocated when None.  Returns (state, bias_out)."""
    E = bias.shape[0]
    n_pool = sum(int(m.shape[0]) for m in microbatches)
    state = state or EQBState(E, bias.device)
    if keys is None:
        keys = torch.empty(n_pool, E, dtype=torch.int16, device=bias.device)
    if bias_out is None:
        bias_out = torch.empty_like(bias)
    row = 0
    first = True
    for m in microbatches:
        n = int(m.shape[0])
        if n == 0:
            continue  # issues no work
        # every microbatch after the first continues the batch on this stream
        route = qb_route_hist_hi if first else qb_route_hist_hi_next
        route(m, bias, k, state.hist_hi, keys_out=keys[row:row + n], stream=stream)
        first = False
        row += n
    r = rank(n_pool, E, k)
    qb_select_hi(state.hist_hi, r, state.sel, state.r_lo, stream=stream)
    qb_keys_hist_lo(keys, state.sel, state.hist_lo, stream=stream)
    qb_finalize(state.hist_hi, state.hist_lo, state.sel, state.r_lo, bias_out, qkey_out=state.qkey,
                reset=reset, stream=stream)
    return state, bias_out
