"""GB300-native quantile balancing (QB / EQB / K3 / LEI) for MoE routers.

The compute path is the C-ABI library ``libqb.so`` (hand-written sm_103a CUDA
kernels, built from ``csrc/``).  ``exact_distributed_quantiles_gb300.qb`` is
the thin ctypes binding with the same entry-point names; it raises if the
library has not been built.  ``inputs`` draws the seeded synthetic workloads.
Submodules are imported on demand (``from exact_distributed_quantiles_gb300
import qb``), so importing the package itself loads no native code.
"""
