"""CPU fp64 oracle (test infrastructure only; see dsv4sa_oracle's docstring)."""
from .dsv4sa_oracle import *  # noqa: F401,F403
from .dsv4sa_oracle import (e4m3_decode, bf16_decode, kv_rows, index_keys, index_query,  # noqa: F401
                            indexer_logits_row, indexer_logits, topk_row, window_indices,
                            compress_indices, n_visible, sink_softmax_attention, gather_rows,
                            sparse_attn_row, sparse_attn, decode_step, SOFTMAX_SCALE_512)
