"""GB300 (sm_103a) block-batched MXFP4 mixture-of-experts layer.

The compute lives in the CUDA library ``_moe_gb300.so`` (sources in ``csrc/``,
C ABI in ``include/moe.h``); ``binding`` marshals arguments to it and
``layer.MoeLayer`` holds one layer's device buffers.  Importing the package
does not load the library; the first call does, and fails loudly if it has not
been built.
"""

__all__ = ["binding", "layer", "build"]
