"""B300-native (sm_103a) Multi-head Latent Attention decode.

The compute path is the C-ABI library libmla.so (include/mla.h, sources in
csrc/); ``mla`` is its Python binding and ``synth`` draws seeded inputs.
Nothing here computes the method on the CPU.
"""

__all__ = ["build", "mla", "synth"]
