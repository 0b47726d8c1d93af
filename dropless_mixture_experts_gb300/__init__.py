"""GB300-native dropless, sorted-dispatch mixture-of-experts layer.

The compute path is the C-ABI library ``libmoe_gb300.so`` (hand-written CUDA
for sm_103a, built in-tree by ``dropless_mixture_experts_gb300.build``).  The
Python side only marshals arguments: ``abi`` exposes the C entry points under
their own names and ``layer`` composes them into a forward pass and a train
step.  Importing this package does not load the library; the first call into
``abi`` does, and raises if the library has not been built.
"""

from .synthetic import CONFIGS, MoEConfig, make_inputs  # noqa: F401

__all__ = ["CONFIGS", "MoEConfig", "make_inputs"]
