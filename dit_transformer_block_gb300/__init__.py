"""GB300-native forward pass of one joint audio-video DiT block.

The compute lives in the C-ABI library ``libh3block.so`` (hand-written sm_103a
kernels); ``dit_transformer_block_gb300.h3`` is its thin ctypes binding. The
library is loaded on first use of the binding, so importing the package (for
example for ``inputs``) does not need a GPU.
"""
__all__ = ["inputs", "h3"]
