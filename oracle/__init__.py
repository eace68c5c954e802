"""Float64 CPU oracle of the single-token RoPE + GQA decode step.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs
of ``bench.py`` may call it. It shares no code with the CUDA path.

It is the plain definition written out with numpy in float64: rotate q and the
new k, write k and v into the cache slot, gather the logical K and V, expand the
KV heads with repeat-interleave, then softmax(q K^T / sqrt(D)) V with a
max-subtracted two-pass softmax. No blocking, no online softmax, no splits.

Pages cited (by title and section):

* [KVC-GQA-RoPE] "Transformer推理核心：KV Cache、GQA与RoPE原理与工程实践"
  (§2 autoregressive decoding and the KV cache, §2.1 attention formula and the
  decode shapes, §2.2 GQA and repeat_interleave, §3 RoPE, §4.1 cache layout and
  paging, §5.1 the per-layer decode step, §5.3 debugging checks).
* [SelfAttn-Step] "4. 自注意力机制推理：单步计算、KV Cache的引入与原理"
  (§4.1 attention formula, §4.3 the KV cache, §4.5 preallocated cache written by
  index and the single-step pseudo-code).
* [Opt-2026] "Transformer架构优化实战2026：注意力机制、KV Cache与推理加速完整指南"
  (§二 standard attention, §三 FlashAttention's default 1/sqrt(d_k) scale, §四
  KVCache.update / PagedKVCache / the cache-size formula, §六 GQA and n_rep).

``oracle.quant`` adds the INT8 KV cache with per-head scales and a bf16 window of
recent tokens ([KVC-GQA-RoPE] §4.3), and ``oracle.verify`` the multi-query decode of a
speculative-verify step (gamma new tokens, causal inside the chunk; [Opt-2026] §五), each
with its readings stated in its header.

Parity status: every function here is pinned by tests that do not retype it
(library routines, complex-number rotation, brute force, closed forms and the
pages' worked numbers); none is "parity unpinned".
"""

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits, f64_to_storage, storage_to_f64  # noqa: F401
from .rope import inv_freq, rope_angles, apply_rope  # noqa: F401
from .kvcache import (append_contiguous, append_paged, logical_kv_contiguous,  # noqa: F401
                      logical_kv_paged, kv_cache_bytes)
from .attention import (repeat_kv, softmax, attention, gqa_decode_attention,  # noqa: F401
                        causal_attention)
from .decode import decode_step  # noqa: F401
from . import quant  # noqa: F401
from . import verify  # noqa: F401
