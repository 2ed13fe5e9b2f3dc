"""GB300 (sm_103a) RMSNorm for training, and LayerNorm beside it: a C-ABI CUDA library plus
a thin torch binding.

The CUDA library is loaded lazily on the first call; importing the package needs no GPU
(so the input generator ``synth`` is usable on any host).  There is no CPU fallback.
"""
from .layernorm import LayerNormTrain, layernorm_bwd, layernorm_fwd, layernorm_train  # noqa: F401
from .ops import (RMSNormTrain, rmsnorm_bwd, rmsnorm_bwd_recompute, rmsnorm_fwd,  # noqa: F401
                  rmsnorm_train)

__all__ = ["rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_bwd_recompute", "rmsnorm_train", "RMSNormTrain",
           "layernorm_fwd", "layernorm_bwd", "layernorm_train", "LayerNormTrain"]
