"""Absorbed Multi-head Latent Attention on the latent KV cache, for GB300 (sm_103a).

The hot path lives in libmla.so (hand-written CUDA, C ABI in include/mla.h);
``binding`` marshals PyTorch tensors into it, ``pipeline`` chains the steps,
``workloads`` draws the seeded synthetic inputs.
"""
from .binding import (MLAError, declared_symbols, library_path, load_library, make_dims,  # noqa: F401
                      mla_absorb_q, mla_attn_decode, mla_attn_decode_q8_0, mla_attn_decode_static,
                      mla_attn_prefill, mla_attn_prefill_materialized, mla_attn_prefill_materialized_q8_0,
                      mla_prefill_materialized_workspace_size,
                      mla_attn_prefill_q8_0, mla_decode_workspace_size, mla_prefill_workspace_size, mla_get_device_error,
                      mla_late_decompress, mla_late_decompress_f16, mla_convert_bf16_to_f16, mla_output_project, mla_quantize_q8_0, mla_rope_append, mla_selftest_wait_timeout,
                      mla_status_string,
                      mla_version)
from .pipeline import mla_decode, mla_prefill, mla_prefill_projected  # noqa: F401
