"""Benchmark of the QB hot path on the full-step workload.

Workload (one step): 48 MoE router layers, each with 16 microbatches of 32768
tokens (524288 tokens per layer), E = 256 experts, top-6, fp32 logits
N(0,1) + per-expert offset N(0,0.5) with a 10% skew towards 16 experts per
microbatch; per layer: EQB hi pass (sigmoid, top-7, margins, BF16 keys, hi-
byte histogram), rank select, lo pass over the stored keys, finalize (exact
quantile, centering, bias update in place, histogram reset), then LEI with
eta = 8e-5 on an fp32 score gradient [524288, 256] per 32768-token local
batch.  Shapes follow the testbed of "Exact Quantile Balancing and Load-Error
Injection for Mixture-of-Experts" (256 routed experts, top-6, 48 MoE layers;
eta = 8e-5).  Inputs are synthetic and seeded (data: "synthetic").

Metric: routed tokens per second per layer = layers * tokens per layer / step
time.  48 GiB of inputs stay resident in HBM, far larger than L2, so no L2
flush is needed between steps.

``--impl reference`` times the CPU oracle (the plain restatement of the
method) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "QB routed tokens/s per layer (E=256,k=6, 2-pass EQB) on 1 GB300; % of HBM roofline"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one hi-pass
# launch (route256_kernel, keys written, no top-k output) on a 524288-token
# layer, from an ncu capture of that launch.  Reported only while the
# kernel's sources hash to the value they had when the counters were taken.
ROUTE_TRAFFIC = {"sha1": "9caf9b404b8e9a128ce7dfb04ff503deabad3269", "tokens": 524288,
                 "bytes": (537.010432 + 232.794368) * 1e6}
ROUTE_SOURCES = ("qb_route256.cuh", "qb_route256_f32.cu", "qb_route.cuh", "qb_device.cuh")
# Warp instructions of the same capture (smsp__inst_executed.sum), for the
# issue-rate roofline of this issue-bound kernel; same hash guard.
ROUTE_INSTR = {"tokens": 524288, "warp_instructions": 126612727}
# Warp instructions (smsp__inst_executed.sum) of one K3 microbatch of 65536
# bf16 tokens: the alpha pass (route256_kernel, K3 mode) plus the count
# kernel, from an ncu capture of those launches; reported while the K3
# sources hash to the value they had when it was taken.
K3_INSTR = {"sha1": "afc61768ab95c5de323af2ba864056ba75218ff8", "tokens": 65536,
            "warp_instructions": 12850624 + 13207384}
K3_SOURCES = ("qb_route256.cuh", "qb_route256_bf16.cu", "qb_route.cuh", "qb_device.cuh",
              "qb_k3.cu")
UNIT = "tokens/s/layer"
WORKLOAD = "full_step"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def _sources_sha1(files) -> str:
    import hashlib
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, "exact_distributed_quantiles_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _route_sources_match() -> bool:
    return _sources_sha1(ROUTE_SOURCES) == ROUTE_TRAFFIC["sha1"]


def _issue_peak():
    """Warp-instruction issue peak: SMs x 4 schedulers x 1 instruction per
    cycle x the maximum SM clock (MEASURED_PEAKS.json's, else 2070 MHz)."""
    try:
        mhz = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 4 * mhz * 1e6


def _route_traffic(tokens: int):
    import hashlib
    h = hashlib.sha1()
    for f in ROUTE_SOURCES:
        with open(os.path.join(ROOT, "exact_distributed_quantiles_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != ROUTE_TRAFFIC["sha1"]:
        return None
    return ROUTE_TRAFFIC["bytes"] * tokens / ROUTE_TRAFFIC["tokens"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return 6800.0, "fallback", {"bf16_tflops": 1900.0}


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) >= 9:
                for i, n in enumerate(names):
                    if r[5 + i].lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


# --------------------------------------------------------------------------- GPU arm

class FullStep:
    def __init__(self, qb, inputs, device, layers: int, seed_offset: int = 0):
        self.qb = qb
        w = inputs.WORKLOADS[WORKLOAD]
        self.w = w
        self.L = layers
        E, k, n = w.E, w.k, w.n_pool
        dev = device
        self.logits = torch.empty(layers, n, E, dtype=torch.float32, device=dev)
        self.grads = torch.empty(layers, n, E, dtype=torch.float32, device=dev)
        self.bias = torch.empty(layers, E, dtype=torch.float32, device=dev)
        for l in range(layers):
            b, _ = inputs.router_layer(w, inputs.seed_for(WORKLOAD, l) + seed_offset, device=dev,
                                       out=self.logits[l])
            self.bias[l].copy_(b)
            inputs.score_grad(w, inputs.seed_for(WORKLOAD, l) + seed_offset, n_tokens=n,
                              device=dev, out=self.grads[l])
        self.hist_hi = torch.zeros(layers, E, 256, dtype=torch.int32, device=dev)
        self.hist_lo = torch.zeros(layers, E, 256, dtype=torch.int32, device=dev)
        self.sel = torch.zeros(layers, E, dtype=torch.int32, device=dev)
        self.r_lo = torch.zeros(layers, E, dtype=torch.int32, device=dev)
        # top-k sets and LEI workspaces alternate between layers: a layer's
        # LEI finishes while the next layer routes
        self.keys = torch.empty(n, E, dtype=torch.int16, device=dev)
        self.topk = [torch.empty(n, k, dtype=torch.int32, device=dev) for _ in range(2)]
        self.ws = [torch.empty(w.n_micro, E, dtype=torch.float32, device=dev) for _ in range(2)]
        self.side = torch.cuda.Stream(device=dev)
        self.ev_hi = [torch.cuda.Event() for _ in range(2)]
        self.ev_rho = [torch.cuda.Event() for _ in range(2)]
        self.pending = None  # (grad, slot) of a layer whose grad update is still to be enqueued
        self.R = qb.rank(n, E, k)
        self.launches_per_layer = {"eqb": 4, "lei": 2}
        self.hi_events = []

    def layer(self, l, logits=None, grad=None, lei=True, time_hi=False, join=False,
              per_microbatch=False):
        """One layer.  EQB runs on the current stream.  LEI needs only this
        layer's top-k sets: its rho kernel runs on a second stream beside the
        EQB tail, and its grad update is enqueued right behind the NEXT
        layer's hi pass as a programmatic dependent (lei_apply_overlap), so
        that the bulk-copy unit streams the gradient while that pass routes.
        join=True (or flush()) enqueues the pending grad update at once."""
        qb, w = self.qb, self.w
        j = l & 1
        main = torch.cuda.current_stream()
        lg = self.logits[l] if logits is None else logits
        prev = self.pending
        if prev is not None:
            main.wait_event(self.ev_rho[prev[1]])  # its eta*rho is in the workspace
        if time_hi:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
        # the top-k sets are LEI's input only: EQB alone does not produce them
        if per_microbatch:
            # one hi-pass call per 32768-token microbatch, as they would arrive
            # (each after the first continues the batch: qb_route_hist_hi_next)
            n = w.n_tokens
            for m in range(w.n_micro):
                sl = slice(m * n, (m + 1) * n)
                route = qb.qb_route_hist_hi if m == 0 else qb.qb_route_hist_hi_next
                route(lg[sl], self.bias[l], w.k, self.hist_hi[l], keys_out=self.keys[sl],
                      topk_out=self.topk[j][sl] if lei else None)
        else:
            qb.qb_route_hist_hi(lg, self.bias[l], w.k, self.hist_hi[l], keys_out=self.keys,
                                topk_out=self.topk[j] if lei else None)
        if time_hi:
            e1.record()
            self.hi_events.append((e0, e1))
        if prev is not None:
            if time_hi:  # (not behind the timed pass)
                qb.lei_apply(prev[0], self.ws[prev[1]], batch_tokens=w.n_tokens)
            else:
                qb.lei_apply_overlap(prev[0], self.ws[prev[1]], batch_tokens=w.n_tokens)
            self.pending = None
        self.ev_hi[j].record(main)
        if lei:
            self.side.wait_event(self.ev_hi[j])
            with torch.cuda.stream(self.side):
                qb.lei_rho(self.topk[j], w.E, w.eta, self.ws[j], batch_tokens=w.n_tokens)
            self.ev_rho[j].record(self.side)
            self.pending = (self.grads[l] if grad is None else grad, j)
        qb.qb_select_hi(self.hist_hi[l], self.R, self.sel[l], self.r_lo[l])
        qb.qb_keys_hist_lo(self.keys, self.sel[l], self.hist_lo[l])
        qb.qb_finalize(self.hist_hi[l], self.hist_lo[l], self.sel[l], self.r_lo[l], self.bias[l],
                       reset=True)
        if join:
            self.flush()

    def flush(self):
        """Enqueue the pending grad update (the last layer's) on the current stream."""
        if self.pending is not None:
            g, j = self.pending
            main = torch.cuda.current_stream()
            main.wait_event(self.ev_rho[j])
            self.qb.lei_apply(g, self.ws[j], batch_tokens=self.w.n_tokens)
            self.pending = None

    def step(self, lei=True, time_hi=False, per_microbatch=False):
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        for l in range(self.L):
            self.layer(l, lei=lei, time_hi=time_hi, per_microbatch=per_microbatch)
        self.flush()
        main.wait_stream(self.side)


def _timed(fn, steps, warmup, dist_on):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if dist_on:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    if dist_on:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms


def _per_call_ms(fn, reps, warmup):
    """Mean device time of one fn() over reps back-to-back calls (CUDA events)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _graph(fn):
    """fn captured once as a CUDA graph (after one eager call, which sets the
    kernels' attributes); returns its replay."""
    fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            fn()
    torch.cuda.current_stream().wait_stream(cs)
    _graph.keep.append(graph)
    return graph.replay


_graph.keep = []


def _rotating(replays):
    """One call = the next of the given replays, in turn."""
    it = [0]

    def f():
        replays[it[0] % len(replays)]()
        it[0] += 1
    return f


def k3_component(qb, inputs, dev, reps, warmup, peak_hbm):
    """K3 histogram mode: E=256, k=8, 4 x 65536 bf16 tokens, 1000 bins; one
    global batch = four k3_route_hist calls + k3_finalize.  Four copies of the
    batch at distinct addresses (512 MiB together) are used in turn so that L2
    holds none of them."""
    w3 = inputs.WORKLOADS["k3"]
    bias3, mbs3 = inputs.router_layer(w3, inputs.seed_for("k3"), device=dev)
    copies = [[m.clone() for m in mbs3] for _ in range(4)]
    bounds = inputs.k3_initial_bounds(bias3).to(dev)
    hist3 = torch.zeros(w3.E, 1000, dtype=torch.int32, device=dev)
    # two alpha buffers in turn: a chained call's alpha pass may overlap the
    # previous call's counting
    alpha3 = torch.empty(2, w3.n_tokens, dtype=torch.float32, device=dev)
    b3 = bias3.clone()
    R3 = qb.rank(w3.n_pool, w3.E, w3.k)

    def k3_hist_only(c, chained=True):
        for i, m in enumerate(copies[c]):
            f = qb.k3_route_hist_next if chained and i else qb.k3_route_hist
            f(m, b3, w3.k, bounds, hist3, alpha3[i % 2])

    def k3_batch(c):
        k3_hist_only(c)
        qb.k3_finalize(hist3, R3, bounds, b3, reset=True)

    # each call shape captured as CUDA graphs (one per copy of the batch), so
    # that the times are the device's, not the host's launch rate
    ms_batch = _per_call_ms(_rotating([_graph(lambda c=c: k3_batch(c)) for c in range(4)]),
                            reps, warmup)
    ms_hist = _per_call_ms(_rotating([_graph(lambda c=c: k3_hist_only(c)) for c in range(4)]),
                           reps, warmup)
    ms_hist_w = _per_call_ms(_rotating([_graph(lambda c=c: k3_hist_only(c, False))
                                        for c in range(4)]), reps, warmup)
    qb.qb_zero_i32(hist3)
    k3_bytes = w3.n_pool * w3.E * 2  # bf16 logits read once (algorithmic)
    return {
        "workload": "k3: 4x65536 bf16 tokens, E=256, k=8, 1000 bins",
        "value": w3.n_pool / (ms_batch / 1e3), "unit": "tokens/s", "ms_per_batch": ms_batch,
        "launches_per_batch": 2 * w3.n_micro + 1, "cuda_graph": True,
        "microbatches_chained": True, "hist_ms_per_batch_each_waiting": ms_hist_w,
        "roofline": {"bound": "hbm", "kernel": "k3_route_hist (route256_kernel alpha pass + k3_count_kernel)",
                     "achieved": k3_bytes / (ms_hist / 1e3) / 1e9, "peak": peak_hbm,
                     "unit": "GB/s", "frac": k3_bytes / (ms_hist / 1e3) / 1e9 / peak_hbm,
                     "bytes_per_batch": k3_bytes, "hist_ms_per_batch": ms_hist},
        # both K3 passes are bound by instruction issue, not by HBM
        "roofline_issue": (None if K3_INSTR["warp_instructions"] is None
                           or _sources_sha1(K3_SOURCES) != K3_INSTR["sha1"] else {
            "bound": "alu", "kernel": "k3_route_hist (route256_kernel alpha pass + k3_count_kernel)",
            "achieved": K3_INSTR["warp_instructions"] * w3.n_pool / K3_INSTR["tokens"]
            / (ms_hist / 1e3), "peak": _issue_peak(), "unit": "warp instructions/s",
            "frac": K3_INSTR["warp_instructions"] * w3.n_pool / K3_INSTR["tokens"]
            / (ms_hist / 1e3) / _issue_peak()})}


def gemm_component(qb, inputs, dev, reps, warmup, peak_hbm, peaks):
    """Router GEMM front end: 4 x 32768 tokens of bf16 hidden states [., 2048]
    x W [2048, 256]; one global batch = four GEMM + hi-pass calls, select, lo
    pass over the stored keys, finalize.  Its 512 MiB of hidden states exceed
    L2."""
    w5 = inputs.WORKLOADS["router_gemm"]
    bias5, W, hs = inputs.gemm_layer(w5, inputs.seed_for("router_gemm"), device=dev)
    w_t = W.t().contiguous()
    n, E, H = w5.n_tokens, w5.E, w5.hidden
    logits5 = torch.empty(n, E, dtype=torch.float32, device=dev)
    keys5 = torch.empty(w5.n_pool, E, dtype=torch.int16, device=dev)
    hi5 = torch.zeros(E, 256, dtype=torch.int32, device=dev)
    lo5 = torch.zeros(E, 256, dtype=torch.int32, device=dev)
    sel5 = torch.zeros(E, dtype=torch.int32, device=dev)
    rlo5 = torch.zeros(E, dtype=torch.int32, device=dev)
    b5 = bias5.clone()
    R5 = qb.rank(w5.n_pool, E, w5.k)

    def gemm_only():
        for h in hs:
            qb.qb_router_gemm(h, w_t, logits5)

    def fused_calls(chained=True):
        # the fused path: logits stay in tensor memory (no logits_out); the
        # microbatches after the first continue the batch (..._next)
        for i, h in enumerate(hs):
            f = qb.qb_router_gemm_hist_hi_next if chained and i else qb.qb_router_gemm_hist_hi
            f(h, w_t, b5, w5.k, None, hi5, keys_out=keys5[i * n:(i + 1) * n])

    def gemm_batch():
        fused_calls()
        qb.qb_select_hi(hi5, R5, sel5, rlo5)
        qb.qb_keys_hist_lo(keys5, sel5, lo5)
        qb.qb_finalize(hi5, lo5, sel5, rlo5, b5, reset=True)

    # CUDA graphs of each call shape (device times, not the host's launch rate)
    ms5 = _per_call_ms(_graph(gemm_batch), reps, warmup)
    ms_g = _per_call_ms(_graph(gemm_only), reps, warmup)
    # per microbatch, the 4 microbatches in turn (none of them in L2); and
    # with every call waiting for the one before it
    ms_f = _per_call_ms(_graph(fused_calls), reps, warmup) / len(hs)
    ms_fw = _per_call_ms(_graph(lambda: fused_calls(False)), reps, warmup) / len(hs)
    qb.qb_zero_i32(hi5)
    flops = 2.0 * w5.n_pool * H * E
    gbytes = w5.n_pool * H * 2 + H * E * 2 * w5.n_micro + w5.n_pool * E * 4
    tflops = flops / (ms_g / 1e3) / 1e12
    gbs = gbytes / (ms_g / 1e3) / 1e9
    peak_tc = peaks.get("bf16_tflops")
    # the fused kernel the path runs (gemm_route_kernel): per microbatch it
    # reads the hidden states and W^T and writes the uint16 keys (the logits
    # stay in tensor memory), and does the GEMM's flops
    f_flops = 2.0 * n * H * E
    f_bytes = n * H * 2 + H * E * 2 + n * E * 2
    f_tflops = f_flops / (ms_f / 1e3) / 1e12
    f_gbs = f_bytes / (ms_f / 1e3) / 1e9
    # its bound is whichever floor is higher: about 226 FLOP per HBM byte
    # here, below the ridge (peak TFLOP/s / peak GB/s, about 283), so HBM
    f_hbm_bound = peak_tc is None or f_bytes / (peak_hbm * 1e9) >= f_flops / (peak_tc * 1e12)
    return {
        "workload": "router_gemm: 4x32768 tokens, hidden 2048 bf16 x W [2048,256] bf16 on the "
                    "tensor cores with the EQB hi pass (k=6) in the GEMM epilogue, then select, "
                    "lo pass, finalize",
        "value": w5.n_pool / (ms5 / 1e3), "unit": "tokens/s", "ms_per_batch": ms5,
        "launches_per_batch": w5.n_micro + 3,
        "fused_ms_per_microbatch": ms_f,
        "fused_ms_per_microbatch_each_waiting": ms_fw,
        "roofline": {"bound": "hbm" if f_hbm_bound else "tensor",
                     "kernel": "gemm_route_kernel (tcgen05 GEMM + hi pass in the epilogue; "
                               "keys written, logits kept in tensor memory)",
                     "achieved": f_gbs if f_hbm_bound else f_tflops,
                     "peak": peak_hbm if f_hbm_bound else peak_tc,
                     "unit": "GB/s" if f_hbm_bound else "TFLOP/s",
                     "frac": f_gbs / peak_hbm if f_hbm_bound else f_tflops / peak_tc,
                     "bytes_per_microbatch": f_bytes, "flops_per_microbatch": f_flops,
                     "tensor_tflops": f_tflops,
                     "tensor_frac": f_tflops / peak_tc if peak_tc else None,
                     "hbm_gbs": f_gbs, "hbm_frac": f_gbs / peak_hbm},
        # the plain GEMM (logits written) for comparison
        "plain_gemm": {"ms_per_batch": ms_g, "bytes_per_batch": gbytes, "flops_per_batch": flops,
                       "tensor_tflops": tflops,
                       "tensor_frac": tflops / peak_tc if peak_tc else None,
                       "hbm_gbs": gbs, "hbm_frac": gbs / peak_hbm}}


def rank_average_component(qb, inputs, dev, reps, warmup, peak_hbm):
    """Rank-averaged QB on the pooled workload (E=256, k=6, 8 x 16384 skewed
    tokens) as 8 ranks of one microbatch each: per rank the EQB steps on its
    own tokens, then the average of the 8 selected keys.  Timed next to the
    pooled EQB of the same tokens."""
    w = inputs.WORKLOADS["eqb_pooled"]
    bias, mbs = inputs.router_layer(w, inputs.seed_for("eqb_pooled"), device=dev)
    E, n = w.E, w.n_tokens
    keys = torch.empty(w.n_pool, E, dtype=torch.int16, device=dev)
    hi = torch.zeros(E, 256, dtype=torch.int32, device=dev)
    lo = torch.zeros_like(hi)
    sel = torch.empty(E, dtype=torch.int32, device=dev)
    r_lo = torch.empty_like(sel)
    qk = torch.empty(w.n_micro, E, dtype=torch.int16, device=dev)
    scratch = torch.empty(E, dtype=torch.float32, device=dev)
    out = torch.empty(E, dtype=torch.float32, device=dev)

    def ranks():
        for p, m in enumerate(mbs):
            kp = keys[p * n:(p + 1) * n]
            qb.qb_route_hist_hi(m, bias, w.k, hi, keys_out=kp)
            qb.qb_select_hi(hi, qb.rank(n, E, w.k), sel, r_lo)
            qb.qb_keys_hist_lo(kp, sel, lo)
            qb.qb_finalize(hi, lo, sel, r_lo, scratch, qkey_out=qk[p], reset=True)
        qb.qb_rank_average(qk, out)

    def pooled():
        for p, m in enumerate(mbs):
            qb.qb_route_hist_hi(m, bias, w.k, hi, keys_out=keys[p * n:(p + 1) * n])
        qb.qb_select_hi(hi, qb.rank(w.n_pool, E, w.k), sel, r_lo)
        qb.qb_keys_hist_lo(keys, sel, lo)
        qb.qb_finalize(hi, lo, sel, r_lo, out, reset=True)

    ms_r = _per_call_ms(ranks, reps, warmup)
    ms_p = _per_call_ms(pooled, reps, warmup)
    return {"workload": "eqb_pooled as 8 ranks: 8 x 16384 tokens, E=256, k=6",
            "value": w.n_pool / (ms_r / 1e3), "unit": "tokens/s", "ms_per_batch": ms_r,
            "pooled_eqb_ms_per_batch": ms_p, "launches_per_batch": 4 * w.n_micro + 1,
            "roofline": {"bound": "hbm", "bytes_per_batch": w.n_pool * E * 8,
                         "achieved": w.n_pool * E * 8 / (ms_r / 1e3) / 1e9, "peak": peak_hbm,
                         "unit": "GB/s",
                         "frac": w.n_pool * E * 8 / (ms_r / 1e3) / 1e9 / peak_hbm}}


def maxvio_component(qb, inputs, dev, reps, warmup):
    """MaxVio of one full-step layer: 524288 tokens' top-6 sets in 16 local
    batches of 32768 (the sets the hi pass writes for LEI)."""
    w = inputs.WORKLOADS["full_step"]
    topk = inputs.random_topk(w.n_pool, w.E, w.k, seed=4, device=dev)
    loads = torch.empty(w.n_micro, w.E, dtype=torch.int32, device=dev)
    mv = torch.empty(2, dtype=torch.float64, device=dev)
    ms = _per_call_ms(lambda: qb.qb_maxvio(topk, w.E, loads, mv, batch_tokens=w.n_tokens),
                      reps, warmup)
    nbytes = w.n_pool * w.k * 4
    return {"workload": "full_step layer: 16 x 32768 tokens, top-6 of 256", "ms_per_call": ms,
            "launches_per_call": 2, "bytes_per_call": nbytes,
            "achieved_gbs": nbytes / (ms / 1e3) / 1e9}


def components(qb, inputs, dev, reps, warmup, peak_hbm, peaks):
    """The other timed paths: K3 histogram mode, the router-GEMM front end,
    rank-averaged QB and the MaxVio diagnostic."""
    return {"k3": k3_component(qb, inputs, dev, reps, warmup, peak_hbm),
            "router_gemm": gemm_component(qb, inputs, dev, reps, warmup, peak_hbm, peaks),
            "rank_average": rank_average_component(qb, inputs, dev, reps, warmup, peak_hbm),
            "maxvio": maxvio_component(qb, inputs, dev, reps, warmup)}


def cpu_baseline_sample(n_tokens: int, layer: int = 0, threads: int | None = None):
    """Oracle on a bounded sample: n_tokens of one full-step layer through the
    two-pass EQB of the headline metric (route by full sort, keys, hi/lo
    counts, exact select by sort, centering).  threads: OpenMP threads for the
    oracle (None: all cores).  Returns (seconds, tokens, threads used)."""
    import oracle
    from exact_distributed_quantiles_gb300 import inputs
    oracle.build()
    w = inputs.WORKLOADS[WORKLOAD]
    ws = inputs.scaled(w, n_micro=max(1, n_tokens // w.n_tokens),
                       n_tokens=min(n_tokens, w.n_tokens))
    bias, mbs = inputs.router_layer(ws, inputs.seed_for(WORKLOAD, layer))
    mbs_np = [m.numpy() for m in mbs]
    b_np = bias.numpy()
    all_cores = oracle.num_threads()
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        used = oracle.num_threads()
        t0 = time.perf_counter()
        oracle.eqb_global_batch(mbs_np, b_np, ws.k)
        dt = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(all_cores)
    return dt, ws.n_pool, used


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n_tok = args.ref_tokens
    for _ in range(args.warmup):
        cpu_baseline_sample(n_tok)
    times = []
    cores = 1
    for _ in range(args.steps):
        dt, n, cores = cpu_baseline_sample(n_tok)
        times.append(dt)
    tot = sum(times)
    value = args.steps * n_tok / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: 48 layers x 16x32768 tokens, E=256, k=6; reference "
                               f"arm times the CPU oracle on {n_tok} tokens of layer 0 per step",
                   "sample_tokens_per_step": n_tok},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n_tok} tokens of full-step layer 0: EQB (full-sort routing, "
                                   "keys, counts, sort select, centering)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--ref-tokens", type=int, default=32768)
    ap.add_argument("--cpu-tokens", type=int, default=524288)
    ap.add_argument("--cpu-tokens-single", type=int, default=65536)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-components", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every kernel from the host instead of replaying the step "
                         "captured once as a CUDA graph")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, "k3", "router_gemm", "rank_average", "maxvio"],
                    help="full_step (the headline line: EQB step, with LEI in full_step) or one "
                         "of the other timed paths alone")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    torch.cuda.set_device(local)
    if dist_on:
        torch.distributed.init_process_group("nccl")
    from exact_distributed_quantiles_gb300 import build, inputs
    build.build()
    from exact_distributed_quantiles_gb300 import qb

    if args.workload != WORKLOAD:
        peak, peak_kind, peaks = _peaks()
        dev = torch.device("cuda", local)
        reps = max(args.steps, 10)
        if args.workload == "k3":
            c = k3_component(qb, inputs, dev, reps, args.warmup, peak)
        elif args.workload == "router_gemm":
            c = gemm_component(qb, inputs, dev, reps, args.warmup, peak, peaks)
        elif args.workload == "rank_average":
            c = rank_average_component(qb, inputs, dev, reps, args.warmup, peak)
        else:
            c = maxvio_component(qb, inputs, dev, reps, args.warmup)
        if rank == 0:
            print(json.dumps({"workload": args.workload, "n_gpus": world, "steps": reps,
                              "warmup": args.warmup, "data": "synthetic", **c}), flush=True)
        if dist_on:
            torch.distributed.destroy_process_group()
        return

    fs = FullStep(qb, inputs, torch.device("cuda", local), args.layers, seed_offset=rank * 100)
    w = fs.w
    tokens_layer_step = fs.L * w.n_pool  # token-layers per step per rank

    # full step (EQB + LEI), by default replayed from a CUDA graph captured
    # once (every replay launches every kernel of the 48 layers again; the
    # bias and histograms are updated in place, as in training)
    def graphed(fn):
        if args.no_graph:
            return fn
        fn()  # first calls outside the capture (kernel attributes)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            with torch.cuda.graph(graph, stream=cs):
                fn()
        torch.cuda.current_stream().wait_stream(cs)
        graphs.append(graph)
        return graph.replay

    graphs = []
    # the headline: the two-pass EQB step (per layer: hi pass over the layer's
    # 16 microbatches, select, lo pass over the keys, finalize = bias update
    # and histogram reset)
    eqb_fn = graphed(lambda: fs.step(lei=False))
    with ClockSampler(local) as clk:
        ms_eqb = _timed(eqb_fn, args.steps, args.warmup, dist_on)
    # the hi-pass launches of the same EQB step, one event pair around each
    fs.hi_events.clear()
    ms_hi_loop = _timed(lambda: fs.step(lei=False, time_hi=True), 1, 0, dist_on)
    hi_ms = [a.elapsed_time(b) for a, b in fs.hi_events]
    # the full step of the workload: EQB + LEI (eta=8e-5) per 32768-token batch
    ms = _timed(graphed(lambda: fs.step(lei=True)), args.steps, args.warmup, dist_on)
    # the EQB step with the hi pass called once per 32768-token microbatch
    ms_eqb_mb = _timed(graphed(lambda: fs.step(lei=False, per_microbatch=True)), args.steps,
                       args.warmup, dist_on)
    ms_step = ms / args.steps
    full_value = world * tokens_layer_step / (ms_step / 1e3)
    eqb_value = world * tokens_layer_step / ((ms_eqb / args.steps) / 1e3)

    peak, peak_kind, peaks = _peaks()
    n, E, k = w.n_pool, w.E, w.k
    hi_bytes = n * E * (4 + 2)               # logits read, keys write (EQB needs no top-k)
    hi_avg_ms = statistics.mean(hi_ms) if hi_ms else float("nan")
    eqb_bytes = hi_bytes + n * E * 2                      # hi pass + lo pass over the keys
    # + top-k write (LEI's input), LEI counts read, grad read and write
    step_bytes = eqb_bytes + n * k * 4 + n * k * 4 + n * E * 4 * 2
    achieved = hi_bytes / (hi_avg_ms / 1e3) / 1e9

    # end to end through host buffers: the EQB step with every layer's logits
    # copied in from pinned host memory and its new bias copied out
    e2e = None
    if not args.no_e2e:
        lg_h = fs.logits[0].cpu().pin_memory()
        b_out = torch.empty(fs.L, E, dtype=torch.float32).pin_memory()
        # two device buffers; layer l+1's logits are copied in on one stream
        # and layer l's bias out on another while layer l computes
        d_lg = [torch.empty_like(fs.logits[0]) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        comp = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_step():
            s_in.wait_stream(comp)
            s_out.wait_stream(comp)
            for l in range(fs.L):
                j = l & 1
                with torch.cuda.stream(s_in):
                    if l >= 2:
                        s_in.wait_event(ev_done[j])  # layer l-2 has read this buffer
                    d_lg[j].copy_(lg_h, non_blocking=True)
                    ev_in[j].record(s_in)
                comp.wait_event(ev_in[j])
                fs.layer(l, logits=d_lg[j], lei=False)
                ev_done[j].record(comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[j])
                    b_out[l].copy_(fs.bias[l], non_blocking=True)
            comp.wait_stream(s_out)  # the step ends with its last copy out

        e2e_steps = max(1, min(args.steps, 3))
        ms_e2e = _timed(e2e_step, e2e_steps, 1, dist_on)
        e2e = {"value": world * tokens_layer_step / ((ms_e2e / e2e_steps) / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": fs.L * n * E * 4, "d2h_bytes_per_step": fs.L * E * 4,
               "steps": e2e_steps}

    comps = None
    if not args.no_components:
        comps = components(qb, inputs, fs.logits.device, max(args.steps, 10), args.warmup, peak,
                           peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        dt, nt, cores = cpu_baseline_sample(args.cpu_tokens)
        dt1, nt1, _ = cpu_baseline_sample(args.cpu_tokens_single, threads=1)
        cpu = {"value": nt / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{nt} tokens of full-step layer 0 through the oracle's EQB "
                         "(full-sort routing, keys, counts, sort select, centering) "
                         f"({dt:.1f} s on {cores} threads)",
               "single_thread": {"value": nt1 / dt1, "unit": UNIT, "cores": 1,
                                 "sample": f"{nt1} tokens of the same layer, one thread "
                                           f"({dt1:.1f} s)"}}

    if rank == 0:
        eqb_ms_step = ms_eqb / args.steps
        line = {
            "metric": METRIC, "value": eqb_value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": eqb_ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: {fs.L} layers x {w.n_micro}x{w.n_tokens} tokens, "
                                   f"E={E}, k={k}; a step = per layer the two-pass EQB: hi pass "
                                   "over the layer's 16 microbatches (one call), select, lo pass "
                                   "over the stored keys, finalize (bias update, histogram reset); "
                                   "LEI timed in full_step",
                       "layers": fs.L, "tokens_per_layer": n, "E": E, "k": k,
                       "parallelism": f"replicas x{world} (token shards, no collective)",
                       "cuda_graph": not args.no_graph,
                       "l2": f"resident logits ({fs.L * n * E * 4 / 2**30:g} GiB) larger than L2 "
                             "(129 MB); no flush"},
            # HBM roofline of the EQB step: 2048 algorithmic bytes per token
            # (logits read, keys written and read back)
            "eqb_roofline": {"bytes_per_layer": eqb_bytes,
                             "achieved": eqb_bytes * fs.L / (eqb_ms_step / 1e3) / 1e9,
                             "peak": peak, "unit": "GB/s",
                             "frac": eqb_bytes * fs.L / (eqb_ms_step / 1e3) / 1e9 / peak,
                             "frac_nominal": eqb_bytes * fs.L / (eqb_ms_step / 1e3) / 1e9
                             / NOMINAL_HBM_GBS},
            # the same EQB step with one hi-pass call per 32768-token microbatch
            "eqb_per_microbatch": {
                "value": world * tokens_layer_step / ((ms_eqb_mb / args.steps) / 1e3), "unit": UNIT,
                "ms_per_step": ms_eqb_mb / args.steps, "hi_pass_calls_per_layer": w.n_micro,
                "frac": eqb_bytes * fs.L / ((ms_eqb_mb / args.steps) / 1e3) / 1e9 / peak},
            # the full step of the workload: EQB + LEI (eta = 8e-5) per 32768-token
            # local batch (rho beside the EQB tail, grad update beside the next
            # layer's hi pass)
            "full_step": {"value": full_value, "unit": UNIT, "ms_per_step": ms_step,
                          "gpu_launches_per_step": fs.L * (fs.launches_per_layer["eqb"]
                                                           + fs.launches_per_layer["lei"])},
            "step_roofline": {
                "bytes_per_layer": step_bytes, "eqb_bytes_per_layer": eqb_bytes,
                "achieved": step_bytes * fs.L / (ms_step / 1e3) / 1e9,
                "eqb_achieved": eqb_bytes * fs.L / ((ms_eqb / args.steps) / 1e3) / 1e9,
                "peak": peak, "unit": "GB/s",
                "frac": step_bytes * fs.L / (ms_step / 1e3) / 1e9 / peak,
                "eqb_frac": eqb_bytes * fs.L / ((ms_eqb / args.steps) / 1e3) / 1e9 / peak,
                # the same against GB300's nominal HBM3e bandwidth (8 TB/s)
                "frac_nominal": step_bytes * fs.L / (ms_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "eqb_frac_nominal": eqb_bytes * fs.L / ((ms_eqb / args.steps) / 1e3) / 1e9
                / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "kernel": "qb_route_hist_hi (route256_kernel, keys out, no top-k out)",
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": _route_traffic(n),
                         "bytes_per_launch": hi_bytes, "avg_launch_ms": hi_avg_ms},
            "roofline_issue": (None if ROUTE_INSTR["warp_instructions"] is None
                               or not _route_sources_match() else {
                "bound": "alu", "kernel": "qb_route_hist_hi (route256_kernel, keys out, no top-k out)",
                "achieved": ROUTE_INSTR["warp_instructions"] * n / ROUTE_INSTR["tokens"]
                / (hi_avg_ms / 1e3), "peak": _issue_peak(), "unit": "warp instructions/s",
                "frac": ROUTE_INSTR["warp_instructions"] * n / ROUTE_INSTR["tokens"]
                / (hi_avg_ms / 1e3) / _issue_peak()}),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "components": comps,
            "gpu_launches": args.steps * fs.L * fs.launches_per_layer["eqb"],
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
