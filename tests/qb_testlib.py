"""Helpers shared by the GPU parity tests: run the CUDA path through the C-ABI
binding, fetch results as numpy, and compare with the oracle."""
import numpy as np
import torch


def np_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def host_logits(t: torch.Tensor) -> np.ndarray:
    """Host copy of logits in the oracle's input format (fp32, or bf16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def gpu_route(qb, logits, bias, k, hist=None):
    """One hi pass with every optional output; returns numpy arrays."""
    N, E = logits.shape
    dev = logits.device
    hist = torch.zeros(E, 256, dtype=torch.int32, device=dev) if hist is None else hist
    keys = torch.empty(N, E, dtype=torch.int16, device=dev)
    topk = torch.empty(N, k, dtype=torch.int32, device=dev)
    alpha = torch.empty(N, dtype=torch.float32, device=dev)
    qb.qb_route_hist_hi(logits, bias, k, hist, keys_out=keys, topk_out=topk, alpha_out=alpha)
    torch.cuda.synchronize()
    assert qb.device_status() == 0
    return dict(hist_hi=hist.cpu().numpy(), keys=np_u16(keys), topk=topk.cpu().numpy(),
                alpha=alpha.cpu().numpy())


def assert_route_matches(orc, res, logits_host, bias_host, k):
    ref = orc.route(logits_host, bias_host, k, want=("alpha", "margins", "topk"))
    assert np.array_equal(res["alpha"].view(np.uint32), ref["alpha"].view(np.uint32)), "alpha"
    assert np.array_equal(res["keys"], orc.keys(ref["margins"])), "keys"
    # the GPU writes the top-k set in ascending expert order
    assert np.array_equal(res["topk"], np.sort(ref["topk"], axis=1)), "topk"
    return ref
