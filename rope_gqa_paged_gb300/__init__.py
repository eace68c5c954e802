"""GB300-native single-token RoPE + GQA decode attention (contiguous and paged KV cache).

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI
(include/rra.h, built into lib/librra_gb300.so); this package binds it with ctypes
and uses torch only for device memory and streams.
"""

from .rra import (RRA_BF16, RRA_ERR_BLOCK_ID, RRA_ERR_POSITION, RRA_ERR_SEQ_LEN, RRA_ERR_TIMEOUT,  # noqa: F401
                  RRA_ERR_WORKSPACE,
                  RRA_F32, RraError, lib, lib_path, rra_decode_attn_contig, rra_decode_attn_paged,
                  rra_decode_num_splits, rra_decode_step_contig, rra_decode_step_paged, rra_decode_workspace_bytes,
                  rra_kv_bytes, rra_rope_append,
                  rra_status_str, rra_rope_append_q8, rra_decode_attn_q8, rra_decode_step_q8,
                  rra_decode_q8_num_splits, rra_rope_append_verify, rra_verify_attn, rra_verify_step,
                  rra_verify_num_splits, rra_verify_workspace_bytes, rra_prefill_attn, rra_prefill_step)
from .step import DecodeStep, DecodeStepQ8, PrefillStep, VerifyStep  # noqa: F401
from ._build import build  # noqa: F401
