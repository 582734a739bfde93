"""fp64 CPU oracle for fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never do, and this package imports nothing from them.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants, a brute-force loop,
library special cases and a hand-worked example under ``tests/golden/``);
no function is "parity unpinned".
"""
from .sdpa import (  # noqa: F401
    attention,
    attention_head,
    attention_rows,
    attention_varlen,
    attention_varlen_rows,
    decode,
    decode_multi,
    kv_head_of,
    rope_rotate,
    round_bf16,
    log_sum_exp,
    scores,
    softmax_two_pass,
    to_f64,
    visible_mask,
)
from .brute import attention_loops  # noqa: F401
