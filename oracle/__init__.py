"""fp64 CPU oracle of the KV-cached Talker forward.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py. The CUDA library and its Python binding never
import it, and it never imports them.
"""
from .talker_oracle import (Oracle, OracleCache, rms_norm, rope_neox, silu, softmax,  # noqa: F401
                            attend_one, kv_group, argmax_low, decode_row_lazy_cache,
                            embed_codes, suppress_logits, code_predictor_frame,
                            q8_0_quantize, q8_0_dequantize, q8_0_roundtrip)
