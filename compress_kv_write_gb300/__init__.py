"""GB300 (sm_103a) KV-cache write path for DeepSeek-V4-style serving.

The compute lives in libkvq.so (C ABI in include/kvq.h, CUDA kernels in
csrc/); this package holds its build script, a thin ctypes binding with the
same entry-point names (kvq_store, kvq_compress, kvq_dequant,
kvq_translate_loc) and the seeded synthetic input generators.
"""
from .kvq import (  # noqa: F401
    BF16, F32, FLAG_NORM, FLAG_ROPE, I32, I64, V41, V41_FP4, KVQError, bytes_per_token,
    kvq_compress, kvq_compress_decode, kvq_dequant, kvq_dequant_slots, kvq_store, kvq_translate_loc, lib, page_bytes,
)
