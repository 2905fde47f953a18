"""fp64 CPU oracle for Multi-head Latent Attention decode.

TEST INFRASTRUCTURE, not part of the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import, call or execute anything in this package.  The
CUDA library never links against it and this package imports nothing from
the CUDA side.
"""

from .mla import *  # noqa: F401,F403
