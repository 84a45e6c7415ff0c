"""GB300-native (sm_103a) Qwen3-style RMSNorm forward and backward.

The compute lives in ``librmsnorm.so`` (hand-written CUDA, C ABI declared in
``include/rmsnorm.h``). ``rmsnorm_fwd_bwd_02_gb300.rmsnorm`` is the thin
ctypes binding with the same entry-point names, and
``rmsnorm_fwd_bwd_02_gb300.autograd`` holds the torch.autograd functions and
nn.Modules over it (``RMSNorm``, ``ResidualRMSNorm``). Importing this
package does not load the library, so the seeded input generators in
``workloads`` work on machines without a GPU.
"""
__all__ = ["rmsnorm", "workloads", "autograd"]
