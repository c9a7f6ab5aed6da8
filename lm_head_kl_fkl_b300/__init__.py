"""Fused chunked top-K forward-KL distillation loss for the LM head, native to B300 (sm_103a).

The compute path is the C-ABI library ``libfkl.so`` (tcgen05/TMA kernels); this
package only marshals torch tensors into it.  Importing the package does not
load the library: the first call does, and fails loudly if it is missing.
"""
__all__ = ["forward", "backward", "forward_backward", "mix_forward", "mix_backward", "teacher_topk",
           "fkl_loss", "workspace_size", "FKLError"]


def __getattr__(name):
    if name in __all__ or name in ("FKLLoss", "FKLLossKeepLogits"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
