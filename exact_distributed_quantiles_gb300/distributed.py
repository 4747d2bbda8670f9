"""Data-parallel EQB across ranks: the exchange protocol around the kernels.

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph: each rank histograms the high byte of its margins into 256
bins per expert, one all-reduce locates the bin holding the r-th smallest
value, a second pass histograms the low byte inside that bin, and a second
all-reduce of 256 counts per expert finishes the select -- 2*E*256 int32 per
layer whatever the number of tokens.  "[Dev] Add global-batch quantile
balancing", "Implementation": the counts are summed over the tensor-, data-
and context-parallel ranks, then every rank updates its bias in place.

Every rank runs the same select and finalize on the same summed counts, so
the biases agree bit for bit on every rank and equal the single-process
result on the pooled tokens (partition invariance).

The compute steps come from an ``ops`` object, so the same protocol drives the
CUDA library (``CudaOps``: one rank per GPU, NCCL) and, in tests, any other
implementation with the same five methods over ``gloo``.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class CudaOps:
    """Kernel-backed steps for one rank (device tensors, libqb)."""

    def __init__(self):
        from . import qb
        self.qb = qb

    def zeros_hist(self, E, device):
        return torch.zeros(E, 256, dtype=torch.int32, device=device)

    def route_hist_hi(self, logits, bias, k, hist_hi, keys_out):
        self.qb.qb_route_hist_hi(logits, bias, k, hist_hi, keys_out=keys_out)

    def select_hi(self, hist_hi, r):
        E = hist_hi.shape[0]
        sel = torch.empty(E, dtype=torch.int32, device=hist_hi.device)
        r_lo = torch.empty_like(sel)
        self.qb.qb_select_hi(hist_hi, r, sel, r_lo)
        return sel, r_lo

    def keys_hist_lo(self, keys, sel, hist_lo):
        self.qb.qb_keys_hist_lo(keys, sel, hist_lo)

    def finalize(self, hist_hi, hist_lo, sel, r_lo, bias_out):
        self.qb.qb_finalize(hist_hi, hist_lo, sel, r_lo, bias_out, reset=True)

    def rank(self, n_pool, E, k):
        return self.qb.rank(n_pool, E, k)


def eqb_global_batch(ops, microbatches, bias, k, group=None):
    """One global batch of EQB on this rank's microbatches, pooled over `group`.

    Returns (bias_out, info) where info holds the summed histograms, the
    selected bins and the pooled token count (the same on every rank)."""
    E = bias.shape[0]
    device = bias.device
    n_local = sum(int(m.shape[0]) for m in microbatches)
    keys = torch.empty(n_local, E, dtype=torch.int16, device=device)
    hist_hi = ops.zeros_hist(E, device)
    row = 0
    for m in microbatches:
        n = int(m.shape[0])
        ops.route_hist_hi(m, bias, k, hist_hi, keys[row:row + n])
        row += n
    local_hi = hist_hi.clone()
    # the token count travels with the first exchange (one extra int64)
    n_pool = torch.tensor([n_local], dtype=torch.int64, device=device)
    dist.all_reduce(n_pool, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(hist_hi, op=dist.ReduceOp.SUM, group=group)  # E*256 int32
    n_pool = int(n_pool.item())
    r = ops.rank(n_pool, E, k)
    sel, r_lo = ops.select_hi(hist_hi, r)
    hist_lo = ops.zeros_hist(E, device)
    ops.keys_hist_lo(keys, sel, hist_lo)
    dist.all_reduce(hist_lo, op=dist.ReduceOp.SUM, group=group)  # E*256 int32
    info = dict(hist_hi=hist_hi.clone(), hist_lo=hist_lo.clone(), sel=sel, r_lo=r_lo,
                n_pool=n_pool, local_hist_hi=local_hi)
    bias_out = torch.empty_like(bias)
    ops.finalize(hist_hi, hist_lo, sel, r_lo, bias_out)
    return bias_out, info
