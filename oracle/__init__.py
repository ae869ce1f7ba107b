"""CPU oracle for one denoising step of block-diffusion MoE decoding.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs use it.  It shares no code with
the CUDA library and imports nothing from it.

Everything is plain numpy in float64, written as the definition of each step;
see ``oracle.moe_step`` for the functions and the passages they follow.
Every function here is pinned by ``tests/test_oracle_*.py`` (closed forms,
invariants, brute force and reductions to textbook routines); none is
"parity unpinned".
"""
from .moe_step import *  # noqa: F401,F403
