"""CPU oracle for chunked Q8_0-KV causal prefill attention.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously correct
statement of what the GPU path computes. It exists so that the tests, the
`__graft_entry__.smoke()` check and the CPU-baseline leg of `bench.py` have
something independent to compare against. The product path (the C-ABI library
and its Python binding) never imports it, and it never imports the product
path: the two share no code, headers, tables or helpers.

Precision: the Q8_0 quantiser is defined bit-exactly in IEEE fp32 (the codes
are integers decided in fp32 on both sides); everything in attention is fp64.

Sources (web pages, cited by title and section):
  * "Core Architecture & The 4-Brick Pipeline", §5 "Brick 4: Barrier-Free
    FlashAttention & Dynamic Q8_0 KV Cache", part 2 "Dynamic Q8_0 KV Cache
    Compression" -- the 34-byte block (32 int8 codes + one fp16 scale),
    symmetric 8-bit quantisation, the 46.88 % volume reduction and the causal
    tile-skipping rule.
  * "Out-of-Core Flash Streaming & Speculative Decode (1M Context)", §1 "The
    Context Memory Wall" (KV byte totals), §3 "Chunked FlashAttention: Exact
    Mathematical Derivation" (the per-chunk recurrence, steps 1-6, and the final
    division), §4 "Mode A vs. Mode B" (triangular causal mask for prefill).

Pinning: every function here is checked in tests/test_oracle_pins.py against
values the pages print, closed forms, invariants and brute force; none is
"parity unpinned".
"""

from .q8_0 import (  # noqa: F401
    BLOCK_VALUES, BLOCK_BYTES, ROW_BYTES,
    quantize_blocks, dequantize_blocks, pack_rows, unpack_rows,
    quantize_kv, dequantize_kv, kv_cache_bytes, fp16_kv_cache_bytes,
)
from .attention import (  # noqa: F401
    attention_rows, attention_unchunked, attention_chunked,
    state_init, chunk_step, finalize,
)
