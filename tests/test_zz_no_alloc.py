"""The allocation-free decode entry point, mla_attn_decode_static.

Some callers of this library cannot allocate device memory: plugins running
inside a host engine that owns every device allocation and forbids cudaMalloc,
or callers with no allocator to take a decode workspace from.  For them
mla_attn_decode_static keeps its split-KV partial results in one fixed device
array inside the library instead of a caller-provided workspace.  This test
calls it through the C ABI twice in a row, with different inputs, and checks
each result against mla_attn_decode with an explicit workspace; it also checks
that a request larger than the fixed scratch is refused before any launch.
The file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _case(lengths, seed):
    from mla_latent_kv_lat_gb300 import workloads as W
    x = W.make_inputs("v3_decode_b32", seed=seed, lengths=lengths)
    rng = np.random.default_rng(seed + 100)
    q_lat = torch.from_numpy(W.to_f16(W.normal_f16(rng, (len(lengths), 128, 512)))[1]).view(torch.float16).cuda()
    q_pe = torch.from_numpy(W.to_bf16(x.q_pe)[1]).view(torch.bfloat16).cuda()
    kv = torch.from_numpy(x.kv_rows_bits()).view(torch.bfloat16).cuda()
    return q_lat, q_pe, kv, torch.from_numpy(x.seq_start).cuda(), torch.from_numpy(x.seq_len).cuda(), int(max(lengths))


def test_static_scratch_decode_matches_workspace_decode():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import build
    from tests.gpu_util import TOL_BF16, assert_tol
    build.build()
    mla.load_library()
    assert mla.mla_get_device_error() == 0
    for lengths, seed in (([3000, 777, 4096, 1, 2049], 0), ([16384, 5, 9000, 12000, 64, 300, 1, 16383], 1)):
        q_lat, q_pe, kv, starts, lens, max_len = _case(lengths, seed)
        B = len(lengths)
        ref = torch.empty(B, 128, 512, dtype=torch.float16, device="cuda")
        ws = torch.empty(mla.mla_decode_workspace_size(128, B, max_len), dtype=torch.uint8, device="cuda")
        mla.mla_attn_decode(q_lat, q_pe, kv, starts, lens, max_len, ws, ref)
        out = torch.full((B, 128, 512), float("nan"), dtype=torch.float16, device="cuda")
        mla.mla_attn_decode_static(q_lat, q_pe, kv, starts, lens, max_len, out)
        torch.cuda.synchronize()
        assert mla.mla_get_device_error() == 0
        assert_tol(out.float().cpu().numpy(), ref.float().cpu().numpy(), TOL_BF16, f"static decode {lengths}")
    # 64 sequences at 128 heads need more than 32 MiB of scratch: refused on the host
    need = mla.mla_decode_workspace_size(128, 64, 32768)
    assert need > 32 << 20
    q_lat = torch.zeros(64, 128, 512, dtype=torch.float16, device="cuda")
    q_pe = torch.zeros(64, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_attn_decode_static(q_lat, q_pe, kv, torch.zeros(64, dtype=torch.int64, device="cuda"),
                                   torch.ones(64, dtype=torch.int32, device="cuda"), 32768, q_lat)
    assert e.value.status == -4
