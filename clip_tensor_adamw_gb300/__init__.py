"""clip + AdamW optimizer step on one GB300 (sm_103a): ScaleTensors, ClipGradNorms and AdamWSteps (also over
parameter groups, and both as one fused step), ClipGradNorms fused into the gradients' last write when that write is
an add, and SGD / SGD with momentum over the same lists.

The compute lives in libmica_optim.so (hand-written CUDA kernels behind the C ABI of include/mica_optim.h); this
package is its Python binding. Build the library with ``python -m clip_tensor_adamw_gb300.build``.
"""
from .mica import (GroupIndex, MicaError, TensorList, lib, mica_accumulate_clip_grad_norms,
                   mica_accumulate_grad_sumsq, mica_adamw_steps,
                   mica_adamw_steps_grouped, mica_clip_adamw_step, mica_clip_factor_from_sumsq, mica_clip_grad_norms, mica_grad_sumsq,
                   mica_launch_count, mica_release_cache,
                   mica_scale_tensors, mica_selftest_grid_wait_timeout, mica_selftest_wait_timeout, mica_sgd_steps,
                   mica_sync, mica_work_items)

__all__ = ["GroupIndex", "MicaError", "TensorList", "lib", "mica_accumulate_clip_grad_norms",
           "mica_accumulate_grad_sumsq", "mica_adamw_steps",
           "mica_adamw_steps_grouped",
           "mica_clip_adamw_step", "mica_clip_factor_from_sumsq", "mica_clip_grad_norms", "mica_grad_sumsq",
           "mica_launch_count", "mica_release_cache",
           "mica_scale_tensors", "mica_selftest_grid_wait_timeout", "mica_selftest_wait_timeout", "mica_sgd_steps",
           "mica_sync", "mica_work_items"]
