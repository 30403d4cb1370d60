"""fp64 CPU oracle for relative-position attention -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg import this package; the library never does.
"""
from .relpos_oracle import (MODE_ALIBI, MODE_DEBERTA, MODE_SHAW, MODE_T5, MODE_TXL,  # noqa: F401
                            alibi_attention_key_positions, alibi_logits, attention, attention_backward,
                            deberta_delta,
                            deberta_logits, deberta_naive, index_ids, shaw_index, shaw_logits,
                            shaw_naive, sinusoid, skew, t5_attention_backward, t5_attention_key_positions,
                            t5_bucket, t5_logits, txl_logits)
