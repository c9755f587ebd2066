"""Plain, slow, fp64 CPU oracle for paged KV-cache attention decode.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports this
package, and this package imports nothing from the product. Only the test
suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import or run it.

Every function states the passage of the source pages it follows. The four
pages are cited by title:

* "LLM의 Paged Attention: 메모리 효율성을 극대화하는 방법" (page pool, page
  table, copy-on-write, the 2048/500 waste example).
* "vLLM의 핵심 이해: PagedAttention" (contiguous cache, token/slot table).
* "serving-paged-attention" (the KV-size formula and its worked example,
  16-token blocks, block tables, sharing, copy-on-write, block size,
  8-bit KV).
* "LLM 추론 확장, 품질·비용 절충 필수" (decode is bandwidth bound,
  MHA/MQA/GQA, online softmax with three running variables).

All arrays are numpy. 16-bit floating point values travel as raw ``uint16``
bit patterns and 8-bit values as raw ``uint8`` codes, so that scatter and copy
results can be compared bit for bit; arithmetic is done in float64.
"""

from .accounting import (
    kv_cache_bytes,
    max_concurrent_requests,
    naive_waste_fraction,
    paged_tail_waste_tokens,
    concurrent_capacity,
    naive_vs_paged_bytes,
)
from .ofp8 import e4m3_decode, e4m3_encode
from .paged_attention import (
    F16,
    BF16,
    FP8_E4M3,
    bits_to_f64,
    reshape_and_cache,
    copy_blocks,
    swap_blocks,
    gather_sequence,
    paged_decode,
    paged_decode_partitioned,
    paged_prefill,
)

__all__ = [
    "kv_cache_bytes",
    "max_concurrent_requests",
    "naive_waste_fraction",
    "paged_tail_waste_tokens",
    "concurrent_capacity",
    "naive_vs_paged_bytes",
    "e4m3_decode",
    "e4m3_encode",
    "F16",
    "BF16",
    "FP8_E4M3",
    "bits_to_f64",
    "reshape_and_cache",
    "copy_blocks",
    "swap_blocks",
    "gather_sequence",
    "paged_decode",
    "paged_decode_partitioned",
    "paged_prefill",
]
