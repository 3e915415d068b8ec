"""CPU oracle for the zero-copy MoE route -> dispatch -> expert -> combine path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference arm may import or run anything in
this package.  The product path (the CUDA library and its Python binding)
never imports it and has no CPU fallback.

The oracle is a plain, slow, obviously-correct numpy implementation in fp64 of
what the path computes (module ``oracle.moe``: routing, placement, the plain,
deduplicated and FP8 dispatch layouts, the SwiGLU expert, the combine, the
router GEMM), and of the GEMM + all-to-all workload on the same heap (module
``oracle.linear_a2a``).  It shares no code with the CUDA path; both take their
inputs from the seeded generator module ``moe_synth``.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
against brute force on tiny inputs, closed forms, invariants, an independent
library routine (torch CPU) and hand-worked examples under ``tests/golden/``.  The end-to-end float values have
no printed worked example in the source pages, so beyond those closed forms
and invariants their absolute values are parity-unpinned.
"""
from .moe import (  # noqa: F401
    bf16_bits_to_f64,
    round_f64_to_bf16_bits,
    router_logits,
    route_topk,
    count_experts,
    place_pairs,
    dispatch_rows,
    dedup_tokens,
    dedup_row_source,
    e4m3_decode,
    e4m3_encode,
    e4m3_encode_array,
    token_scale_exp,
    quantize_rows_e4m3,
    dequantize_rows,
    expert_ffn_rows,
    expert_ffn,
    combine,
    scale_rows,
    combine_sum,
    pipeline,
    slot_address,
)
from .linear_a2a import (  # noqa: F401
    linear,
    linear_exact,
    a2a_blocks,
    gemm_a2a,
    shard_gather,
    a2a_gemm,
)
