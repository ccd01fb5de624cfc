"""fp64 CPU oracle for the Gated DeltaNet forward (test infrastructure only)."""
from .oracle import (build, gating, recurrent, decode, gating_scalar,  # noqa: F401
                     transition_product, attention_form, chunked_wy, default_threads)
