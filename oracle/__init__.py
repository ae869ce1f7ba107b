"""CPU oracle for one denoising step of block-diffusion MoE decoding.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs use it.  It shares no code with
the CUDA library and imports nothing from it.

Everything is plain numpy in float64, written as the definition of each step;
see ``oracle.moe_step`` for the functions and the passages they follow.
Every function here is pinned by ``tests/test_oracle_*.py``: the primitives
(router, coreset, SwiGLU, RMSNorm, commit, loop) by closed forms, invariants,
brute force and reductions to library routines; the composed functions
(``lm_logits``, ``block_decode_step``, ``tiny_model_logits``) by
``tests/test_oracle_step.py``, against the same arithmetic written out in
plain loops, zero-weight and one-token-block special cases, and request
independence.  None is "parity unpinned".
"""
from .moe_step import *  # noqa: F401,F403
