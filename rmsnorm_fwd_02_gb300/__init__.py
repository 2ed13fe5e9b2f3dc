"""GB300 (sm_103a) RMSNorm for training: a C-ABI CUDA library plus a thin torch binding.

The CUDA library is loaded lazily on the first call; importing the package needs no GPU
(so the input generator ``synth`` is usable on any host).  There is no CPU fallback.
"""
from .ops import RMSNormTrain, rmsnorm_bwd, rmsnorm_fwd, rmsnorm_train  # noqa: F401

__all__ = ["rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_train", "RMSNormTrain"]
