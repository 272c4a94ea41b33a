"""CPU oracle for verify attention: test infrastructure, never on the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package."""
from .attention_fp64 import (  # noqa: F401
    decode_bf16, decode_e4m3fn, round_to_bf16, verify_attn_oracle, oracle_from_torch,
)
