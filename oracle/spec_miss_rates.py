"""How often a predicted quantile region misses on fresh data (speculative EQB).

TEST INFRASTRUCTURE ONLY: an analysis run on the oracle, not part of the
product path.  It measures what a speculative single-pass EQB would rely on:
"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph (the exact quantile from a hi-byte histogram, then a lo-byte
histogram inside the selected bin).  A speculative first pass would count the
lo bytes near each expert's predicted quantile; an expert whose new quantile
falls outside its predicted region needs the second pass after all.

Setup: one router layer of the full-step workload (its per-expert logit
offsets kept), a new token sample every step, the bias updated by EQB after
each step ("[Dev] Add global-batch quantile balancing", "Quantile estimator":
the bias is the centred per-expert quantile).  Per step it prints how many
experts leave (a) the previous step's hi bin and (b) windows of 256 / 512 /
1024 keys centred on the previous quantile key, and the share of all margins
inside each region (the counting work of the first pass).

    python oracle/spec_miss_rates.py [--micro 16] [--steps 7]
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle as orc  # noqa: E402
from exact_distributed_quantiles_gb300 import inputs as I  # noqa: E402


def _offsets(seed: int, E: int, std: float) -> torch.Tensor:
    """The per-expert logit offsets of router_layer(seed): its first draw."""
    g = torch.Generator()
    g.manual_seed(int(seed))
    return torch.randn(E, generator=g, dtype=torch.float32) * std


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--micro", type=int, default=16, help="32768-token microbatches per step")
    ap.add_argument("--steps", type=int, default=7)
    ap.add_argument("--first-seed", type=int, default=77000)
    a = ap.parse_args()

    w = I.scaled(I.WORKLOADS["full_step"], n_micro=a.micro)
    E, k = w.E, w.k
    layer_seed = I.seed_for("full_step", 0)
    off_layer = _offsets(layer_seed, E, w.offset_std)
    bias = I.router_layer(I.scaled(w, n_micro=0), layer_seed)[0].numpy()
    prev_sel = prev_key = None
    for t in range(a.steps):
        seed = a.first_seed + t
        off_t = _offsets(seed, E, w.offset_std)
        keys = []
        for x in I.router_layer(w, seed)[1]:
            # the same router as the layer: swap this sample's offsets for the layer's
            x = (x - off_t + off_layer).numpy()
            keys.append(orc.keys(orc.route(x, bias, k, want=("margins",))["margins"]))
        n = sum(kk.shape[0] for kk in keys)
        R = orc.rank(n, E, k)
        hist = np.zeros((E, 256), np.int32)
        for kk in keys:
            orc.hist_hi(kk, hist)
        sel, r_lo = orc.select_hi(hist, R)
        hist_lo = np.zeros((E, 256), np.int32)
        for kk in keys:
            orc.hist_lo(kk, sel, hist_lo)
        qkey = (sel.astype(np.int64) << 8) | orc.select_lo(hist_lo, r_lo).astype(np.int64)
        line = f"step {t}:"
        if prev_sel is not None:
            in_bin = hist[np.arange(E), prev_sel].sum() / (n * E)
            line += f" hi bin: {int((sel != prev_sel).sum())} missed, {in_bin:.4f} of margins;"
            for half in (128, 256, 512):
                lo = prev_key - half
                hit = (qkey >= lo) & (qkey < lo + 2 * half)
                inside = sum(((kk.astype(np.int64) >= lo) & (kk.astype(np.int64) < lo + 2 * half)).sum()
                             for kk in keys)
                line += f" {2 * half}-key window: {int((~hit).sum())} missed, {inside / (n * E):.4f};"
        print(line, flush=True)
        prev_sel, prev_key = sel, qkey
        bias = orc.center(orc.key_decode_array(qkey.astype(np.uint16)).astype(np.float64))


if __name__ == "__main__":
    main()
