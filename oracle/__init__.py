"""fp64 CPU oracle (test infrastructure only; see ``oracle.attention``)."""

from .attention import (E4M3_TABLE, e4m3_decode, e4m3_value, gqa_decode, merge_partials,
                        mla_decode, mla_visible_keys, partial_attention, schedule,
                        softmax_attention, sparse_mla_decode, unit_segments)

__all__ = ["E4M3_TABLE", "e4m3_decode", "e4m3_value", "gqa_decode", "merge_partials",
           "mla_decode", "mla_visible_keys", "partial_attention", "schedule",
           "softmax_attention", "sparse_mla_decode", "unit_segments"]
