"""CPU oracle for the DFlash block-diffusion drafting hot path.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg may import anything in this package. The
product path (the CUDA library and its Python binding) never does, and this
package imports nothing from it.

The oracle is a plain, slow, obviously correct NumPy restatement of what the
method computes, in float64, with bf16 rounding (round to nearest, ties to
even) at exactly the tensors the drafter stores or feeds to a matrix product.
See ``oracle.dflash`` for the functions and the passages each one follows.
"""
from .dflash import *  # noqa: F401,F403
