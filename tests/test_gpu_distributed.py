"""The data-parallel EQB protocol driven by the CUDA library (CudaOps).

"Exact Quantile Balancing and Load-Error Injection for Mixture-of-Experts",
EQB paragraph: each rank histograms the high byte of its own margins, one
all-reduce, the select, the lo-byte pass, a second all-reduce.  "[Dev] Add
global-batch quantile balancing", "Validation": rank-local histograms differ,
the reduced histogram matches an independent update, every rank ends with the
same bias.

Every call on this pool has one GPU, so the ranks here share it: (a) one rank
over NCCL, and (b) two processes on the one GPU exchanging over gloo with CUDA
tensors, each routing its own token shard with libqb.  The ranks' kernels
never wait on one another (the exchange is a host-side collective), so
sharing the GPU cannot deadlock them.  Both are compared bit for bit with the
oracle on the pooled tokens.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from exact_distributed_quantiles_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _workload():
    # E = 256 (the specialised routing pass); 6 microbatches with a ragged
    # last tile each, dealt to the ranks in turn
    w = inputs.scaled(inputs.WORKLOADS["eqb_pooled"], n_micro=6, n_tokens=2001)
    bias, mbs = inputs.router_layer(w, 77)
    return w, bias, mbs


def _rank_main(rank, world, port, outdir, backend):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    torch.cuda.set_device(0)
    dist.init_process_group(backend, rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=120))
    from exact_distributed_quantiles_gb300 import distributed, qb
    w, bias, mbs = _workload()
    mine = [m.cuda() for m in mbs[rank::world]]
    b, info = distributed.eqb_global_batch(distributed.CudaOps(), mine, bias.cuda(), w.k)
    torch.cuda.synchronize()
    np.save(os.path.join(outdir, f"bias{rank}.npy"), b.cpu().numpy())
    np.save(os.path.join(outdir, f"local{rank}.npy"), info["local_hist_hi"].cpu().numpy())
    np.save(os.path.join(outdir, f"hi{rank}.npy"), info["hist_hi"].cpu().numpy())
    np.save(os.path.join(outdir, f"lo{rank}.npy"), info["hist_lo"].cpu().numpy())
    np.save(os.path.join(outdir, f"status{rank}.npy"), np.array([qb.device_status()]))
    dist.destroy_process_group()


def _check(tmp_path, orc, world):
    w, bias, mbs = _workload()
    ref = orc.eqb_global_batch([m.numpy() for m in mbs], bias.numpy(), w.k)
    locals_ = []
    for r in range(world):
        assert int(np.load(tmp_path / f"status{r}.npy")[0]) == 0
        b = np.load(tmp_path / f"bias{r}.npy")
        assert np.array_equal(b.view(np.uint32), ref["bias_out"].view(np.uint32))
        assert np.array_equal(np.load(tmp_path / f"hi{r}.npy"), ref["hist_hi"])
        assert np.array_equal(np.load(tmp_path / f"lo{r}.npy"), ref["hist_lo"])
        locals_.append(np.load(tmp_path / f"local{r}.npy"))
    assert np.array_equal(sum(locals_), ref["hist_hi"])
    return locals_


def test_one_rank_over_nccl(tmp_path, orc):
    mp.spawn(_rank_main, args=(1, _free_port(), str(tmp_path), "nccl"), nprocs=1, join=True)
    _check(tmp_path, orc, 1)


def test_two_ranks_on_one_gpu_over_gloo(tmp_path, orc):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path), "gloo"), nprocs=2, join=True)
    l0, l1 = _check(tmp_path, orc, 2)
    assert not np.array_equal(l0, l1)  # rank-local histograms differ before the reduction
