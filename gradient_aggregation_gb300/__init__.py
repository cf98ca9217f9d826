"""GB300-native gradient-aggregation engine.

W simulated workers' fp16 per-layer gradients in one GPU's HBM are fused,
summed in a fixed binary-tree order with fp32 accumulation and a
1/(loss scale x W) unscale, scored by chunk L2 norm, sparsified to the top
fraction of chunks with an fp32 residual, and applied as a momentum-SGD
update of fp32 master weights.  Every step runs in hand-written sm_103a CUDA
kernels behind the C ABI declared in ``include/fc.h``; this package is the
thin Python binding (``gradient_aggregation_gb300.fc``) plus the seeded
workload generator (``gradient_aggregation_gb300.workload``).

Importing the package does not load the CUDA library; the first call into
``fc`` does, and raises if the library has not been built.
"""

__all__ = ["fc", "workload", "build"]
