"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this package.  The library's product
path (the CUDA kernels behind the C ABI) never calls into it, and it shares no
code with that path: the only module both sides use is the seeded input
generator ``exact_io_aware_10_gb300.workloads``, which holds no attention
arithmetic.

Sources (cited per function):
  [FA-notes]  "精读笔记 08：FlashAttention" (llm-papers-study), the study notes on
              the FlashAttention paper: §2.1 standard attention, §3.1 online
              softmax, §3.2 tiling / Algorithm 1, §3.3 recomputation,
              §3.5 IO complexity (Theorem 2 and its worked A100 example).
  [S12]       "S12 FlashAttention" (llminference tutorial): the online-softmax
              loop ("核心思路"), the paged version ("实现"), the
              exp(-inf - -inf) warning, flash-decoding and the exercises.
  [IO-explained] "FlashAttention: IO-aware explained" (shandesong.com):
              recomputation keeps only the row statistics (m, l).

Pinning status: every function here is pinned by tests under ``tests/``
(closed forms, invariants, finite differences, brute force, the pages'
worked numbers) except the S12 simulator's printed trace, which the pages
print only in part ("parity unpinned" for that trace; no function depends
on it).
"""
from .attention import (  # noqa: F401
    to_f64,
    valid_key_mask,
    attention_probs,
    attention_forward,
    attention_forward_rows,
    attention_forward_varlen,
    attention_backward,
    attention_backward_rows,
    attention_backward_varlen,
    streaming_row_forward,
    algorithm1_forward,
    merge_states,
)
from .decode import (  # noqa: F401
    gather_paged_keys,
    paged_decode,
    paged_decode_streaming,
    split_paged_decode,
)
from .paged_prefill import (  # noqa: F401
    chunk_key_mask,
    paged_prefill,
    paged_prefill_rows,
)
from .block_sparse import (  # noqa: F401
    expand_block_mask,
    block_sparse_forward,
)
from .io_model import (  # noqa: F401
    standard_hbm_accesses,
    flash_hbm_accesses,
    materialized_matrix_bytes,
)
