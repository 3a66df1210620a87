"""CPU oracle (test infrastructure only; see loglinear_oracle's header)."""
from .loglinear_oracle import (  # noqa: F401
    backward_direct,
    backward_sampled,
    decay_rows,
    decode_step,
    fenwick_partition,
    forward_chunked,
    forward_direct,
    hier_rows,
    level,
    level_matrix,
    level_row,
    linear_attention_recurrent,
    lssb,
    recurrence,
    states_from_buckets,
)
from .gdn_oracle import (  # noqa: F401
    gated_deltanet_recurrent,
    gdn_decode_step,
    gdn_direct,
    gdn_recurrence,
    gdn_states_from_buckets,
)
