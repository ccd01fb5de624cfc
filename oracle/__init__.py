"""fp64 CPU oracle for the Gated DeltaNet forward (test infrastructure only)."""
from .oracle import (build, gating, recurrent, decode, decode_mtp, decode_bf16_pool, round_bf16,  # noqa: F401
                     gating_scalar, transition_product, attention_form, chunked_wy, default_threads)
