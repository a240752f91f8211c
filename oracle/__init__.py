"""CPU oracle for the decode-attention KV cache.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product package.  It shares no
code with the CUDA path; the only common input is the seeded generator in
kv_cache_decode_flash_gb300/synth.py, which draws numbers and holds none of
the method's arithmetic.

The numeric routines live in kvc_oracle.c (plain C, fp64 unless the
definition is fp32); this file loads them through ctypes and adds the
row-list model of the sequence operations and the state byte format
(model.py).
"""
from .numerics import lib, F16, Q4_0, Q8_0, f16_to_f64, f32_to_f16, q8_0_quantize, q8_0_dequantize, attn, attn_bruteforce
from .numerics import q4_0_quantize, q4_0_dequantize
from .numerics import rope_rotate, rope_shift_q8_0, rope_shift_f16, keydiff_scores, min_window
from .model import OracleCache, ColdStore, STATE_MAGIC, STATE_VERSION, state_size

__all__ = [
    "lib", "F16", "Q4_0", "Q8_0", "q4_0_quantize", "q4_0_dequantize", "f16_to_f64", "f32_to_f16", "q8_0_quantize", "q8_0_dequantize", "attn",
    "attn_bruteforce", "rope_rotate", "rope_shift_q8_0", "rope_shift_f16", "keydiff_scores", "min_window",
    "OracleCache", "ColdStore",
    "STATE_MAGIC", "STATE_VERSION", "state_size",
]
