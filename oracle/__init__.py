"""CPU oracle (test infrastructure only).  See kvs_oracle.py."""
from .kvs_oracle import (  # noqa: F401
    GROUP, WIDTHS, allocate_bits, attention_scores, block_attention, block_lse, channel_weights, chord_slopes,
    dequantize, distortion, fp16_scale_ru, gram, lowrank_error, ner, numerical_rank, quantize_pack,
    rdkv_compress, ridge_values, spectrum, threshold_keep, trizone_decode, unit_rms)
