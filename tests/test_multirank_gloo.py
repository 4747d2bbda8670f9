"""Two-rank EQB over gloo on CPU: the exchange protocol of the data-parallel
path (exact_distributed_quantiles_gb300.distributed), driven by the oracle's
counting steps.

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph: rank-local hi-byte histograms, one all-reduce, the select, the
lo-byte pass, a second all-reduce; the result is the exact pooled quantile
whatever the sharding.  "[Dev] Add global-batch quantile balancing",
"Validation": rank-local histograms differ before the reduction, the reduced
histogram matches an independent quantile update, and every rank ends with
the same bias.  A rank that dies before the second exchange makes the other
rank's collective fail within its timeout instead of hanging.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_distributed_quantiles_gb300 import distributed, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleOps:
    """The five steps of the protocol, computed by the CPU oracle."""

    def __init__(self):
        import oracle
        self.o = oracle

    def zeros_hist(self, E, device):
        return torch.zeros(E, 256, dtype=torch.int32)

    def route_hist_hi(self, logits, bias, k, hist_hi, keys_out):
        m = self.o.route(logits.numpy(), bias.numpy(), k, want=("margins",))["margins"]
        kk = self.o.keys(m)
        keys_out.copy_(torch.from_numpy(kk.view(np.int16)))
        hist_hi += torch.from_numpy(self.o.hist_hi(kk))

    def select_hi(self, hist_hi, r):
        sel, r_lo = self.o.select_hi(hist_hi.numpy(), r)
        return torch.from_numpy(sel), torch.from_numpy(r_lo)

    def keys_hist_lo(self, keys, sel, hist_lo):
        hist_lo += torch.from_numpy(self.o.hist_lo(keys.numpy().view(np.uint16), sel.numpy()))

    def finalize(self, hist_hi, hist_lo, sel, r_lo, bias_out):
        lo = self.o.select_lo(hist_lo.numpy(), r_lo.numpy())
        qkey = ((sel.numpy().astype(np.int64) << 8) | lo).astype(np.uint16)
        q = self.o.key_decode_array(qkey).astype(np.float64)
        bias_out.copy_(torch.from_numpy(self.o.center(q)))

    def rank(self, n_pool, E, k):
        return self.o.rank(n_pool, E, k)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _workload():
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], E=64, k=6, n_micro=4, n_tokens=600)
    bias, mbs = inputs.router_layer(w, 2024)
    return w, bias, mbs


def _rank_main(rank, world, port, outdir, die_early):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    w, bias, mbs = _workload()
    mine = mbs[rank::world]  # this rank's microbatches (a token shard)
    ops = OracleOps()
    if die_early and rank == 1:
        os._exit(3)  # the rank disappears before any exchange
    try:
        b, info = distributed.eqb_global_batch(ops, mine, bias, w.k)
        np.save(os.path.join(outdir, f"bias{rank}.npy"), b.numpy())
        np.save(os.path.join(outdir, f"local{rank}.npy"), info["local_hist_hi"].numpy())
        np.save(os.path.join(outdir, f"hi{rank}.npy"), info["hist_hi"].numpy())
        np.save(os.path.join(outdir, f"lo{rank}.npy"), info["hist_lo"].numpy())
    except Exception as e:  # a peer vanished: the collective raised instead of hanging
        with open(os.path.join(outdir, f"error{rank}.txt"), "w") as f:
            f.write(type(e).__name__)
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def test_two_rank_eqb_matches_pooled_oracle(tmp_path, orc):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path), False), nprocs=2, join=True)
    b0 = np.load(tmp_path / "bias0.npy")
    b1 = np.load(tmp_path / "bias1.npy")
    assert np.array_equal(b0.view(np.uint32), b1.view(np.uint32))  # identical on every rank
    w, bias, mbs = _workload()
    ref = orc.eqb_global_batch([m.numpy() for m in mbs], bias.numpy(), w.k)
    assert np.array_equal(b0.view(np.uint32), ref["bias_out"].view(np.uint32))
    assert np.array_equal(np.load(tmp_path / "hi0.npy"), ref["hist_hi"])
    assert np.array_equal(np.load(tmp_path / "lo1.npy"), ref["hist_lo"])
    l0, l1 = np.load(tmp_path / "local0.npy"), np.load(tmp_path / "local1.npy")
    assert not np.array_equal(l0, l1)  # rank-local histograms differ before the reduction
    assert np.array_equal(l0 + l1, ref["hist_hi"])


def test_lost_rank_fails_the_exchange_instead_of_hanging(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path), True))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(not p.is_alive() for p in procs)
    assert procs[1].exitcode == 3
    assert (tmp_path / "error0.txt").exists()
    assert not (tmp_path / "bias0.npy").exists()
