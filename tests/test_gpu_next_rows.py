"""Parity of the rows built around the path (through the C ABI) with the CPU
oracle on seeded inputs:

* the output projection after late decompression (the method page, sec. 4:
  the heads' outputs flattened and multiplied by wo, einsum hdD,bhqd->bqD),
  alone and chained after the whole absorbed path.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_lat_gb300 as mla
from mla_latent_kv_lat_gb300 import workloads as W
from oracle import mla_oracle as O
from tests.gpu_util import TOL_BF16, TOL_Q8, Dev, assert_tol, bf16_dev, f16_dev

MLA_ERR_RANGE = -7

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from mla_latent_kv_lat_gb300 import build
    build.build()
    mla.load_library()
    assert mla.mla_get_device_error() == 0


# ---------------------------------------------------------------------------
# Output projection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,T,D", [(16, 1, 64), (16, 77, 2048), (32, 300, 320), (128, 257, 7168), (48, 128, 512)])
def test_output_project_matches_oracle(H, T, D):
    rng = np.random.default_rng(H * 1000 + T)
    o = W.normal_f16(rng, (T, H, 128), 0.5)
    w_o = W.make_wo(H, D, seed=T).astype(np.float16).astype(np.float32)
    u = torch.full((T, D), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_output_project(f16_dev(o), f16_dev(w_o), u)
    got = u.cpu().numpy().astype(np.float64)
    ref = O.output_projection(o, w_o)
    # fp32 accumulation of H*128 exact fp16 x fp16 products
    assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref)) * np.sqrt(H / 16) + 1e-7
    assert mla.mla_get_device_error() == 0


def test_late_decompress_f16_is_the_rounded_fp32_result():
    rng = np.random.default_rng(21)
    T, H = 300, 32
    o_lat = f16_dev(W.normal_f16(rng, (T, H, 512), 0.3))
    wv_b = bf16_dev(W.normal_bf16(rng, (H, 512, 128), 1 / np.sqrt(512)))
    o32 = torch.empty(T, H, 128, dtype=torch.float32, device="cuda")
    o16 = torch.empty(T, H, 128, dtype=torch.float16, device="cuda")
    mla.mla_late_decompress(o_lat, wv_b, o32)
    mla.mla_late_decompress_f16(o_lat, wv_b, o16)
    assert torch.equal(o16, o32.to(torch.float16))      # the same sums, rounded once (nearest even)
    assert mla.mla_get_device_error() == 0


def test_convert_bf16_to_f16_is_exact_and_reports_range():
    rng = np.random.default_rng(22)
    src = bf16_dev(W.normal_bf16(rng, (64, 1000), 0.02))
    src[3, 5] = 0.0
    src[7, 9] = -1.0e-7                              # lands in fp16's subnormal range
    dst = torch.full(src.shape, float("nan"), dtype=torch.float16, device="cuda")
    mla.mla_convert_bf16_to_f16(src, dst)
    assert torch.equal(dst, src.to(torch.float16))
    assert mla.mla_get_device_error() == 0
    src[60, 999] = 1.0e5                             # past fp16's 65504
    mla.mla_convert_bf16_to_f16(src, dst)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE


def _w_o_f16(w_o: np.ndarray) -> torch.Tensor:
    """The model's bf16 w_o converted once to the fp16 the projection takes."""
    w16 = torch.empty(w_o.shape, dtype=torch.float16, device="cuda")
    mla.mla_convert_bf16_to_f16(bf16_dev(w_o), w16)
    return w16


def _projected_chain(x, rows=None):
    w_o = W.make_wo(x.wl.n_head, x.wl.hidden)
    d = Dev(x)
    bufs, pb = mla.mla_prefill_projected(d.q_nope, d.q_pe, d.wk_b, d.wv_b, _w_o_f16(w_o), x.wl.q_pos0, kv=d.kv)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == 0
    sel = np.arange(x.wl.T) if rows is None else rows
    o_ref, _ = O.attention_unabsorbed(x.q_nope[sel], x.q_pe[sel], x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos()[sel],
                                      x.wl.scale)
    return pb.u.cpu().numpy()[sel], O.output_projection(o_ref, w_o)


def test_projected_chain_lite_t4096_every_row():
    got, ref = _projected_chain(W.make_inputs("lite_t4096"))
    assert_tol(got, ref, TOL_BF16, "lite_t4096 u")


def test_projected_chain_v3_chunk_sampled_rows():
    x = W.make_inputs("v3_chunk8192_at32768")
    rows = W.sample_rows(x.wl.T, 512, seed=0, must=(0, 127, 128, x.wl.T - 1))
    got, ref = _projected_chain(x, rows)
    assert_tol(got, ref, TOL_BF16, "v3 chunk u")


# ---------------------------------------------------------------------------
# Materialised prefill (pp_opt): per-head K/V decompressed, standard attention
# ---------------------------------------------------------------------------
def _materialized(x, head_chunk=0, lse=False):
    d = Dev(x)
    T, H = x.wl.T, x.wl.n_head
    o = torch.full((T, H, 128), float("nan"), dtype=torch.float32, device="cuda")
    ls = torch.empty(T, H, dtype=torch.float32, device="cuda") if lse else None
    mla.mla_attn_prefill_materialized(d.q_nope, d.q_pe, d.kv, d.wk_b, d.wv_b, x.wl.q_pos0, o, ls,
                                      head_chunk=head_chunk)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == 0
    return o, ls


@pytest.mark.parametrize("H,T,q_pos0,n_kv,hc", [(16, 256, 0, 256, 0), (16, 100, 37, 200, 0), (32, 1, 0, 1, 0),
                                                (16, 130, 1000, 1200, 5), (128, 33, 300, 333, 64),
                                                (48, 300, 129, 500, 0)])
def test_materialized_prefill_matches_definition(H, T, q_pos0, n_kv, hc):
    x = W.make_inputs("lite_t256", n_head=H, T=T, q_pos0=q_pos0, n_kv=n_kv)
    o, ls = _materialized(x, hc, lse=True)
    ref, ref_lse = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(o.cpu().numpy(), ref, TOL_BF16, "materialized o")
    assert np.max(np.abs(np.expm1(ls.cpu().numpy().astype(np.float64) - ref_lse))) <= 1e-2


def test_materialized_prefill_lite_t4096_every_row():
    x = W.make_inputs("lite_t4096")
    o, _ = _materialized(x)
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(o.cpu().numpy(), ref, TOL_BF16, "materialized lite_t4096 o")


def test_materialized_prefill_v3_chunk_sampled_rows():
    x = W.make_inputs("v3_chunk8192_at32768")
    o, _ = _materialized(x)
    rows = W.sample_rows(x.wl.T, 512, seed=0, must=(0, 127, 128, 4095, 4096, x.wl.T - 1))
    ref, _ = O.attention_unabsorbed(x.q_nope[rows], x.q_pe[rows], x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos()[rows],
                                    x.wl.scale)
    assert_tol(o.cpu().numpy()[rows], ref, TOL_BF16, "materialized v3 chunk o")


def test_materialized_prefill_is_causal_and_chunking_invariant():
    x = W.make_inputs("lite_t256", n_head=32, T=200, q_pos0=100, n_kv=400)
    d = Dev(x)
    o1 = torch.empty(200, 32, 128, dtype=torch.float32, device="cuda")
    o2 = torch.empty_like(o1)
    mla.mla_attn_prefill_materialized(d.q_nope, d.q_pe, d.kv, d.wk_b, d.wv_b, 100, o1)
    d.kv[300:] = float("nan")                     # rows past the last query's position are never read
    mla.mla_attn_prefill_materialized(d.q_nope, d.q_pe, d.kv, d.wk_b, d.wv_b, 100, o2, head_chunk=7)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == 0
    # each head's keys and values do not depend on the other heads: chunking changes nothing
    assert torch.equal(o1, o2)


def _q8_dev(x):
    codes, scales = O.quantize_q8_0(np.concatenate([x.c_kv, x.k_pe], axis=1))
    deq = O.dequantize_q8_0(codes, scales)
    return torch.from_numpy(codes).cuda(), torch.from_numpy(np.ascontiguousarray(scales.T)).cuda(), deq


@pytest.mark.parametrize("H,T,q_pos0,n_kv,hc", [(16, 200, 57, 300, 0), (128, 40, 1000, 1100, 32)])
def test_materialized_prefill_q8_matches_definition(H, T, q_pos0, n_kv, hc):
    x = W.make_inputs("v3_q8_chunk8192_at90112", n_head=H, T=T, q_pos0=q_pos0, n_kv=n_kv)
    kv_q, kv_d, deq = _q8_dev(x)
    d = Dev(x)
    o = torch.full((T, H, 128), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_attn_prefill_materialized_q8_0(d.q_nope, d.q_pe, kv_q, kv_d, d.wk_b, d.wv_b, q_pos0, o, head_chunk=hc)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == 0
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, deq[:, :512], deq[:, 512:], x.wk_b, x.wv_b, x.q_pos(),
                                    x.wl.scale)
    assert_tol(o.cpu().numpy(), ref, TOL_Q8, "materialized q8 o")


def test_materialized_prefill_q8_chunk_sampled_rows():
    x = W.make_inputs("v3_q8_chunk8192_at90112")
    kv_q, kv_d, deq = _q8_dev(x)
    d = Dev(x)
    o = torch.empty(x.wl.T, 128, 128, dtype=torch.float32, device="cuda")
    mla.mla_attn_prefill_materialized_q8_0(d.q_nope, d.q_pe, kv_q, kv_d, d.wk_b, d.wv_b, x.wl.q_pos0, o)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == 0
    rows = W.sample_rows(x.wl.T, 512, seed=0, must=(0, 127, 128, x.wl.T - 1))
    ref, _ = O.attention_unabsorbed(x.q_nope[rows], x.q_pe[rows], deq[:, :512], deq[:, 512:], x.wk_b, x.wv_b,
                                    x.q_pos()[rows], x.wl.scale)
    assert_tol(o.cpu().numpy()[rows], ref, TOL_Q8, "materialized q8 chunk o")
