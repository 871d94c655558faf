"""Float64 CPU oracle (test infrastructure only; see ``oracle.attention``)."""
from .attention import (  # noqa: F401
    NEG_INF,
    SoftmaxState,
    attention_dense,
    attention_dense_backward,
    attention_dense_rows,
    attention_split_decode,
    attention_tiled_rowwise,
    attention_tiled_rowwise_backward,
    causal_mask,
    default_scale,
    empty_state,
    merge_states,
    split_bounds,
    state_of_scores,
)
