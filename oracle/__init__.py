"""fp64 CPU oracle for exact attention (test infrastructure only).

This package is the checker, not the product.  Only the test suite, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py``
may import it.  It shares no code with the CUDA path: it imports nothing from
``exact_tiled_attention_07_gb300`` and the CUDA path imports nothing from here.

Sources it restates (cited by page title and section):

* "Lecture 8 · GPU Performance & FlashAttention" (CS324 notes), §5.1 standard
  attention, §5.2 online softmax, §5.3 tiled forward, §5.4 recomputing
  backward and the D identity, §5.7 causal block skipping, §8.1 FA2's deferred
  normalisation, §8.2 multi-query / grouped-query attention (``oracle/gqa.py``) and
  split-KV decoding with the state merge (``oracle/decode.py``), the FP8 forward with block
  quantisation (``oracle/fp8.py``), §5.7 block-sparse and sliding-window masks
  (``oracle/masks.py``), Exercises 1 and 3.
* "Stanford CS336 Lecture 5 close reading: GPUs ... Flash Attention", §7
  (the FA2-order forward loop).
* "FlashAttention and GPU memory" (world.lapla.si explainer), §08 online
  softmax, §09 backward with recomputation.

Functions whose parity is not pinned by anything outside themselves say so in
their docstring ("parity unpinned"); every other function is pinned by a
``-m "not gpu"`` test in ``tests/test_oracle_*.py``.
"""

from .attention import (  # noqa: F401
    attn_fwd64,
    attn_bwd64,
    attn_fwd64_rows,
    attn_bwd64_query_rows,
    attn_stats64,
    attn_bwd64_key_rows,
    probabilities64,
)
from .online_softmax import (  # noqa: F401
    online_softmax_trace,
    merge_states,
    tiled_fwd_fa2_order,
    tiled_fwd_fa1_order,
    tiled_bwd_recompute,
    causal_tiles_visited,
)
from .gqa import kv_head_of, expand_kv, attn_fwd64_gqa, attn_bwd64_gqa  # noqa: F401,E402
from .decode import decode_fwd64, split_kv_states64, merge_splits64, split_bounds  # noqa: F401,E402
from .fp8 import e4m3_round, e4m3_values, quantize_blocks, dequantize_blocks, attn_fwd64_fp8  # noqa: F401,E402
from .masks import (visible_mask, attn_fwd64_masked, attn_bwd64_masked, tiled_fwd_block_sparse,  # noqa: F401,E402
                    blocks_visited)
