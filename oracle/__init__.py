"""CPU oracle of the DSA forward step and its backward (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg
import this package; the CUDA library never does.
"""
from .dsa_oracle import (  # noqa: F401
    additive_mask_row,
    dsa_decode,
    dsa_prefill,
    index_scores,
    index_scores_backward,
    index_scores_row_backward,
    index_scores_row,
    indexer_inputs,
    linear,
    masked_attention_row,
    masked_attention_row_backward,
    paged_to_dense,
    sparse_attention_backward,
    topk_select,
    update_indexer,
)
