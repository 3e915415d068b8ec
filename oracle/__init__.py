"""CPU oracle for the zero-copy MoE route -> dispatch -> expert -> combine path.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm import or run it.  The product path
(the CUDA library and its Python binding) never imports it and has no CPU
fallback.  Plain fp64 numpy (``oracle.moe``: routing, placement, the plain,
deduplicated and FP8 dispatch layouts, the SwiGLU expert, the combine, the
router GEMM; ``oracle.linear_a2a``: the GEMM + all-to-all workload), sharing
no code with the CUDA path.  Pinned by ``tests/test_oracle.py`` (brute force,
closed forms, invariants, torch CPU, hand-worked goldens in ``tests/golden/``);
beyond those pins the end-to-end float values are parity-unpinned, since the
source pages print no worked example.
"""
from .moe import *  # noqa: F401,F403
from .linear_a2a import *  # noqa: F401,F403
