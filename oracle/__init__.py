"""CPU oracle (test infrastructure only): see ``oracle.dsa_oracle``.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package; the library does not.
"""
from .dsa_oracle import (visible_len, index_scores_row, index_scores,
                         topk_select_row, topk, dequantize, attend_row,
                         sparse_attention, sparse_attention_aux, sparse_attention_step)

__all__ = ["visible_len", "index_scores_row", "index_scores", "topk_select_row",
           "topk", "dequantize", "attend_row", "sparse_attention", "sparse_attention_aux",
           "sparse_attention_step"]
