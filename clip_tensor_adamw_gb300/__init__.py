"""clip + AdamW optimizer step on one GB300 (sm_103a): ScaleTensors, ClipGradNorms and AdamWSteps.

The compute lives in libmica_optim.so (hand-written CUDA kernels behind the C ABI of include/mica_optim.h); this
package is its Python binding. Build the library with ``python -m clip_tensor_adamw_gb300.build``.
"""
from .mica import (MicaError, TensorList, lib, mica_adamw_steps, mica_clip_grad_norms, mica_launch_count,
                   mica_release_cache, mica_scale_tensors, mica_sync)

__all__ = ["MicaError", "TensorList", "lib", "mica_adamw_steps", "mica_clip_grad_norms", "mica_launch_count",
           "mica_release_cache", "mica_scale_tensors", "mica_sync"]
