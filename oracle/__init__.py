"""float64 CPU oracle (test infrastructure; see attention_fp64)."""

from .attention_fp64 import (  # noqa: F401
    AttentionGrads,
    attention_backward,
    attention_backward_loops,
    attention_forward,
    attention_loss,
    causal_executed_tile_pairs,
)
