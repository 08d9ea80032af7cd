"""The bench's work units agree with the oracle's accounting of the pages'
quantities (bytes of a cache row, FLOPs of a query-key pair)."""
import numpy as np

import bench
from mla_latent_kv_lat_gb300 import workloads as W
from oracle import mla_oracle as O


def test_attention_flops_per_pair_match_the_absorbed_count():
    for H in (16, 128):
        assert bench.FLOP_PER_PAIR_HEAD * H == O.flops_per_pair_absorbed(H)
    wl = W.WORKLOADS["v3_chunk8192_at32768"]
    x = W.Inputs(wl, *([np.zeros(0)] * 6))
    assert bench.attn_flops(wl, x) == O.causal_pairs(wl.T, wl.q_pos0) * O.flops_per_pair_absorbed(wl.n_head)


def test_decode_bytes_read_each_row_once():
    for name, row in (("v3_decode_b32", O.latent_row_bytes(2)), ("v3_q8_decode_b8", O.q8_0_row_bytes())):
        wl = W.WORKLOADS[name]
        lens = np.full(wl.B, 1000, np.int32)
        x = W.Inputs(wl, *([np.zeros(0)] * 6), seq_len=lens)
        q_o = wl.B * wl.n_head * ((O.KV_LORA_RANK + O.QK_ROPE) + O.KV_LORA_RANK) * 2
        assert bench.decode_bytes(wl, x) == 1000 * wl.B * row + q_o


def test_append_bytes_per_token():
    # c_kv + k_pe in (bf16), int32 position + int64 slot, the bf16 row and the q8_0 row out
    assert bench.APPEND_TOKEN_BYTES == O.latent_row_bytes(2) + 4 + 8 + O.latent_row_bytes(2) + O.q8_0_row_bytes()
    wl = W.WORKLOADS["v3_cache_append_98304"]
    assert bench.append_bytes(wl) == wl.T * bench.APPEND_TOKEN_BYTES
