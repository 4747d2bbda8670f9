"""Plain CPU oracle for bias-based quantile balancing (QB / EQB / K3 / LEI).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``qb_oracle.c`` (plain C, fp32 in program order for
the routing steps whose results decide integer histogram bins, fp64 for the
quantile interpolation, centering and LEI).  This module only builds that
library with gcc, loads it with ctypes and marshals numpy arrays.

Sources, cited by page title and section:
  * "[Dev] Add global-batch quantile balancing" (Megatron-LM PR 6637),
    "Quantile estimator" and "Implementation": scores, alpha, margins,
    per-expert k/E quantile, mean-centering, the K3 uniform 1000-bin histogram
    over [min b - 1, max b + 1], pooling over every microbatch.
  * "Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
    EQB paragraph (two 256-bin byte histograms over order-preserving BF16
    margins give the exact quantile) and LEI paragraph (add eta * rho_e to the
    score gradient of expert e for every token of the local batch).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qb_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``qb_oracle.c`` into ``liboracle.so`` next to it (gcc, OpenMP if available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "qb_oracle.h")))):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-Wall", "-Wextra"]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = base + extra + ["-o", tmp, _SRC, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB_PATH)
            return _LIB_PATH
    raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{r.stderr}")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        F = ctypes.c_float
        sigs = {
            "orc_sigmoid": (F, [F]),
            "orc_sigmoid_array": (None, [P, P, I64]),
            "orc_exp_neg": (F, [F]),
            "orc_exp_coeffs": (None, [P]),
            "orc_bf16_rne": (ctypes.c_uint16, [F]),
            "orc_key": (ctypes.c_uint16, [F]),
            "orc_key_decode": (F, [ctypes.c_uint16]),
            "orc_keys_array": (None, [P, P, I64]),
            "orc_bf16_array": (None, [P, P, I64]),
            "orc_route": (None, [P, P, I64, I, I, P, P, P, P]),
            "orc_route_bf16": (None, [P, P, I64, I, I, P, P, P, P]),
            "orc_rank": (I64, [I64, I, I]),
            "orc_hist_hi": (None, [P, I64, I, P]),
            "orc_hist_lo": (None, [P, I64, I, P, P]),
            "orc_select_hi": (None, [P, I, I64, P, P]),
            "orc_select_lo": (None, [P, I, P, P]),
            "orc_kth_key_sort": (None, [P, I64, I, I64, P]),
            "orc_center": (None, [P, I, P]),
            "orc_k3_hist": (None, [P, I64, I, F, F, I, P]),
            "orc_k3_finalize": (None, [P, I, I, I64, F, F, P, P, P]),
            "orc_lei": (None, [P, P, I64, I, I, F, P, P]),
            "orc_num_threads": (I, []),
            "orc_set_num_threads": (None, [I]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- scalar pieces

def sigmoid(x) -> np.ndarray:
    """Pinned logistic function, element-wise on float32 input."""
    x = _c(x, np.float32)
    out = np.empty_like(x)
    _load().orc_sigmoid_array(_p(x), _p(out), x.size)
    return out


def exp_neg(x: float) -> float:
    return float(_load().orc_exp_neg(float(x)))


def exp_coeffs() -> np.ndarray:
    c = np.zeros(8, np.float32)
    _load().orc_exp_coeffs(_p(c))
    return c


def bf16_rne(r) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    r = _c(r, np.float32)
    out = np.empty(r.shape, np.uint16)
    _load().orc_bf16_array(_p(r), _p(out), r.size)
    return out


def keys(r) -> np.ndarray:
    """Order-preserving EQB keys of RN_bf16(r) (uint16), -0 folded to +0."""
    r = _c(r, np.float32)
    out = np.empty(r.shape, np.uint16)
    _load().orc_keys_array(_p(r), _p(out), r.size)
    return out


def key_decode(key: int) -> float:
    return float(_load().orc_key_decode(int(key)))


def key_decode_array(k) -> np.ndarray:
    k = np.asarray(k, np.uint16)
    h = np.where(k & 0x8000, k ^ 0x8000, k ^ 0xFFFF).astype(np.uint32) << 16
    return h.view(np.float32)


def rank(n_pool: int, E: int, k: int) -> int:
    """R = ceil(k * n_pool / E), computed in integers."""
    return int(_load().orc_rank(int(n_pool), int(E), int(k)))


# --------------------------------------------------------------------------- routing

def route(logits, bias, k: int, want=("alpha", "scores", "margins", "topk")) -> dict:
    """Per-token routing by full sort.

    ``logits`` is float32 [N,E], or uint16 [N,E] holding bf16 bit patterns.
    Returns a dict with the requested arrays: alpha [N] f32, scores [N,E] f32,
    margins [N,E] f32, topk [N,k] int32 (order: v descending, index ascending).
    """
    lib = _load()
    bias = _c(bias, np.float32)
    is_bf16 = np.asarray(logits).dtype == np.uint16
    logits = _c(logits, np.uint16 if is_bf16 else np.float32)
    N, E = logits.shape
    assert bias.shape == (E,)
    out = {}
    if "alpha" in want:
        out["alpha"] = np.empty(N, np.float32)
    if "scores" in want:
        out["scores"] = np.empty((N, E), np.float32)
    if "margins" in want:
        out["margins"] = np.empty((N, E), np.float32)
    if "topk" in want:
        out["topk"] = np.empty((N, k), np.int32)
    fn = lib.orc_route_bf16 if is_bf16 else lib.orc_route
    fn(_p(logits), _p(bias), N, E, k, _p(out.get("alpha")), _p(out.get("scores")),
       _p(out.get("margins")), _p(out.get("topk")))
    return out


# --------------------------------------------------------------------------- EQB pieces

def hist_hi(key_arr, hist=None) -> np.ndarray:
    key_arr = _c(key_arr, np.uint16)
    N, E = key_arr.shape
    if hist is None:
        hist = np.zeros((E, 256), np.int32)
    _load().orc_hist_hi(_p(key_arr), N, E, _p(hist))
    return hist


def hist_lo(key_arr, sel, hist=None) -> np.ndarray:
    key_arr = _c(key_arr, np.uint16)
    sel = _c(sel, np.int32)
    N, E = key_arr.shape
    if hist is None:
        hist = np.zeros((E, 256), np.int32)
    _load().orc_hist_lo(_p(key_arr), N, E, _p(sel), _p(hist))
    return hist


def select_hi(hist, R: int):
    hist = _c(hist, np.int32)
    E = hist.shape[0]
    sel = np.empty(E, np.int32)
    r_lo = np.empty(E, np.int32)
    _load().orc_select_hi(_p(hist), E, int(R), _p(sel), _p(r_lo))
    return sel, r_lo


def select_lo(hist, r_lo) -> np.ndarray:
    hist = _c(hist, np.int32)
    r_lo = _c(r_lo, np.int32)
    E = hist.shape[0]
    lo = np.empty(E, np.int32)
    _load().orc_select_lo(_p(hist), E, _p(r_lo), _p(lo))
    return lo


def kth_key(key_arr, R: int) -> np.ndarray:
    key_arr = _c(key_arr, np.uint16)
    n, E = key_arr.shape
    q = np.empty(E, np.uint16)
    _load().orc_kth_key_sort(_p(key_arr), n, E, int(R), _p(q))
    return q


def center(q) -> np.ndarray:
    q = _c(q, np.float64)
    out = np.empty(q.shape, np.float32)
    _load().orc_center(_p(q), q.size, _p(out))
    return out


def eqb_global_batch(microbatches, bias, k: int) -> dict:
    """Exact quantile balancing over one global batch.

    ``microbatches``: list of logits arrays [N_m, E] (float32, or uint16 bf16
    bits), all routed with the same ``bias``.  Follows the definition: the
    k/E quantile of each expert's BF16-rounded margins pooled over every
    microbatch is the R-th smallest key (R = ceil(k*N_pool/E)) found by a full
    sort; the hi/lo histograms are direct counts; the new bias is the decoded
    quantile minus the fp64 mean over experts.
    """
    bias = _c(bias, np.float32)
    E = bias.shape[0]
    key_list = []
    for lg in microbatches:
        m = route(lg, bias, k, want=("margins",))["margins"]
        key_list.append(keys(m))
    all_keys = np.concatenate(key_list, axis=0)
    n_pool = all_keys.shape[0]
    R = rank(n_pool, E, k)
    h_hi = np.zeros((E, 256), np.int32)
    for kk in key_list:
        hist_hi(kk, h_hi)
    sel, r_lo = select_hi(h_hi, R)
    h_lo = np.zeros((E, 256), np.int32)
    for kk in key_list:
        hist_lo(kk, sel, h_lo)
    lo = select_lo(h_lo, r_lo)
    qkey = kth_key(all_keys, R)
    # Internal consistency: the two-byte select must land on the sorted answer.
    assert np.array_equal(sel, (qkey >> 8).astype(np.int32)), "hi-byte select disagrees with sort"
    assert np.array_equal(lo, (qkey & 0xFF).astype(np.int32)), "lo-byte select disagrees with sort"
    q = key_decode_array(qkey).astype(np.float64)
    return dict(R=R, n_pool=n_pool, hist_hi=h_hi, hist_lo=h_lo, sel=sel, r_lo=r_lo, lo=lo,
                qkey=qkey, q=q, bias_out=center(q), keys=key_list)


# --------------------------------------------------------------------------- K3

def k3_hist(margins, lo: float, hi: float, nbins: int, hist=None) -> np.ndarray:
    margins = _c(margins, np.float32)
    N, E = margins.shape
    if hist is None:
        hist = np.zeros((E, nbins), np.int32)
    _load().orc_k3_hist(_p(margins), N, E, float(np.float32(lo)), float(np.float32(hi)),
                        int(nbins), _p(hist))
    return hist


def k3_finalize(hist, R: int, lo: float, hi: float):
    hist = _c(hist, np.int32)
    E, nbins = hist.shape
    b = np.empty(E, np.float32)
    bounds = np.empty(2, np.float32)
    q = np.empty(E, np.float64)
    _load().orc_k3_finalize(_p(hist), E, nbins, int(R), float(np.float32(lo)),
                            float(np.float32(hi)), _p(b), _p(bounds), _p(q))
    return b, bounds, q


def k3_global_batch(microbatches, bias, k: int, bounds, nbins: int = 1000) -> dict:
    """K3 histogram quantile balancing over one global batch (approximate)."""
    bias = _c(bias, np.float32)
    E = bias.shape[0]
    lo, hi = np.float32(bounds[0]), np.float32(bounds[1])
    h = np.zeros((E, nbins), np.int32)
    n_pool = 0
    for lg in microbatches:
        m = route(lg, bias, k, want=("margins",))["margins"]
        k3_hist(m, lo, hi, nbins, h)
        n_pool += m.shape[0]
    R = rank(n_pool, E, k)
    b, new_bounds, q = k3_finalize(h, R, lo, hi)
    return dict(R=R, n_pool=n_pool, hist=h, bias_out=b, bounds_out=new_bounds, q=q)


# --------------------------------------------------------------------------- LEI

def lei(grad, topk, eta: float, E: int | None = None):
    """Load-error injection on one local batch; returns (new_grad, load, rho)."""
    g = np.array(grad, dtype=np.float32, copy=True, order="C")
    topk = _c(topk, np.int32)
    N, k = topk.shape
    if E is None:
        E = g.shape[1]
    load = np.empty(E, np.int64)
    rho = np.empty(E, np.float64)
    _load().orc_lei(_p(g), _p(topk), N, E, k, float(np.float32(eta)), _p(load), _p(rho))
    return g, load, rho


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ------------------------------------------------------------ rank-averaged QB

def rank_averaged_qb(rank_microbatches, bias, k: int) -> dict:
    """Rank-averaged QB: each rank's own k/E quantile, averaged over the ranks.

    "Exact Quantile Balancing and Load-Error Injection for Mixture-of-
    Experts", opening paragraph: the MARIN implementation averages rank-local
    quantiles, so its result depends on how the batch is sharded (quantiles do
    not commute with averaging).  Reading used: rank p's quantile q_p[j] is
    the exact order statistic of its own BF16 margins at R_p = ceil(k*N_p/E)
    (what the pooled method computes on that rank's tokens alone); the bias is
    avg[j] = (sum over p in rank order of q_p[j], fp64) / P, then centred like
    the pooled method.  ``rank_microbatches``: one list of logits arrays per
    rank, all routed with ``bias``.
    """
    per_rank = [eqb_global_batch(mbs, bias, k) for mbs in rank_microbatches]
    E = np.asarray(bias).shape[0]
    s = np.zeros(E, np.float64)
    for r in per_rank:
        s = s + r["q"]
    avg = s / float(len(per_rank))
    return dict(q_rank=np.stack([r["q"] for r in per_rank]),
                qkey_rank=np.stack([r["qkey"] for r in per_rank]), avg=avg,
                bias_out=center(avg))


# ---------------------------------------------------------------------- MaxVio

def maxvio(topk_batches, E: int) -> dict:
    """Load imbalance of the routed top-k sets.

    Same paper, testbed paragraph: MaxVio is how far the busiest expert
    exceeds uniform load.  Reading used: for a set of tokens with total n*k
    assignments, T = n*k/E and MaxVio = (max_e load_e - T) / T; "global" over
    all local batches together, "local" the mean over local batches of each
    batch's own value (fp64 throughout).  ``topk_batches``: one int array
    [n_b, k] per local batch.
    """
    loads = [np.bincount(np.asarray(t).ravel(), minlength=E).astype(np.int64) for t in topk_batches]
    tot = np.zeros(E, np.int64)
    for l in loads:
        tot = tot + l
    n_all = sum(int(np.asarray(t).size) for t in topk_batches)
    T = n_all / E
    glob = (float(tot.max()) - T) / T
    loc = 0.0
    for t, l in zip(topk_batches, loads):
        Tb = int(np.asarray(t).size) / E
        loc = loc + (float(l.max()) - Tb) / Tb
    loc = loc / len(topk_batches)
    return dict(loads=np.stack(loads), global_maxvio=glob, local_maxvio=loc)
