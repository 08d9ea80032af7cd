"""Device-side checks of the CUDA path, through the C ABI:

* fp16 range: a bf16 value (cache row, q_pe), an fp32 result (q_lat) or a
  q8_0 block scale that fp16 cannot hold is reported as MLA_ERR_RANGE in the
  device error word, never silently turned into inf or NaN downstream;
* the decode's sequence table: a sequence that names rows outside the cache,
  an empty one or one longer than max_len is skipped and reported as
  MLA_ERR_INVALID_ARG, and the other sequences still match the oracle;
* host buffers with the copies overlapped (pipeline.HostOverlap, the bench's
  end-to-end leg): every step's output equals the plain device call's.

Every case stays inside the allocated tensors (a sequence that runs past the
cache's n_rows still ends inside the buffer), so none can fault even if a
check were broken.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_lat_gb300 as mla
from mla_latent_kv_lat_gb300 import workloads as W
from oracle import mla_oracle as O
from tests.gpu_util import TOL_BF16, TOL_Q8, Dev, assert_tol, bf16_dev, f16_dev

pytestmark = pytest.mark.gpu

MLA_ERR_INVALID_ARG, MLA_ERR_RANGE = -1, -7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from mla_latent_kv_lat_gb300 import build
    build.build()
    mla.load_library()
    assert mla.mla_get_device_error() == 0


def _q8_dev(rows: np.ndarray):
    codes, scales = O.quantize_q8_0(rows)
    return torch.from_numpy(codes).cuda(), torch.from_numpy(np.ascontiguousarray(scales.T)).cuda()


# ---------------------------------------------------------------------------
# fp16 range
# ---------------------------------------------------------------------------
def test_large_cache_value_is_reported_by_prefill():
    x = W.make_inputs("lite_t256", T=64, n_kv=64)
    d = Dev(x)
    d.kv[17, 100] = 1.0e5                          # bf16 1e5 > 65504
    mla.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, 0, kv=d.kv)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE
    d.kv[17, 100] = 1.0
    mla.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, 0, kv=d.kv)
    assert mla.mla_get_device_error() == 0


def test_large_q_pe_is_reported_by_prefill():
    x = W.make_inputs("lite_t256", T=64, n_kv=64)
    d = Dev(x)
    d.q_pe[5, 3, 7] = -2.0e5
    mla.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, 0, kv=d.kv)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE


def test_absorbed_query_past_fp16_is_reported():
    # q_lat = q_nope . wk_b with one q_nope row scaled by 1e5: |q_lat| reaches
    # ~1e5 x |wk_b row sums|, far past 65504
    x = W.make_inputs("lite_t256", T=32, n_kv=32)
    q_nope = x.q_nope.copy()
    q_nope[9, 2] *= 1.0e5
    q_lat = torch.empty(32, 16, 512, dtype=torch.float16, device="cuda")
    assert np.abs(O.absorb_q(q_nope, x.wk_b)).max() > 65504
    mla.mla_absorb_q(bf16_dev(q_nope), bf16_dev(x.wk_b), q_lat)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE
    mla.mla_absorb_q(bf16_dev(x.q_nope), bf16_dev(x.wk_b), q_lat)
    assert mla.mla_get_device_error() == 0


def test_large_cache_value_is_reported_by_decode():
    x = W.make_inputs("v3_decode_b32", n_head=32, lengths=[300, 900])
    d = Dev(x)
    d.kv[1000, 3] = 7.0e4
    mla.mla_decode(d.q_nope, d.q_pe, d.wk_b, d.wv_b, d.seq_start, d.seq_len, 900, kv=d.kv)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE


def test_large_q8_scale_is_reported_by_q8_prefill_and_decode():
    # a block whose largest value is 7e4 gets the scale 7e4 / 127 > 516:
    # 127 x scale does not fit in fp16
    x = W.make_inputs("v3_decode_b32", n_head=16, lengths=[200, 333])
    rows = np.concatenate([x.c_kv, x.k_pe], axis=1)
    rows[250, 40] = 7.0e4
    rows = W.to_bf16(rows)[0]
    kv_q, kv_d = _q8_dev(rows)
    d = Dev(x)
    mla.mla_decode(d.q_nope, d.q_pe, d.wk_b, d.wv_b, d.seq_start, d.seq_len, 333, kv_q=kv_q, kv_d=kv_d)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE
    xp = W.make_inputs("lite_t256", T=16, q_pos0=300, n_kv=533)
    dp = Dev(xp)
    mla.mla_prefill(dp.q_nope, dp.q_pe, dp.wk_b, dp.wv_b, 300, kv_q=kv_q, kv_d=kv_d)
    assert mla.mla_get_device_error() == MLA_ERR_RANGE


# ---------------------------------------------------------------------------
# The decode's sequence table
# ---------------------------------------------------------------------------
def _decode_lat(d: Dev, q_lat, kv_rows, max_len, q8=None):
    B, H = q_lat.shape[0], q_lat.shape[1]
    o_lat = torch.zeros(B, H, 512, dtype=torch.float16, device="cuda")
    ws = torch.empty(mla.mla_decode_workspace_size(H, B, max_len), dtype=torch.uint8, device="cuda")
    if q8 is None:
        mla.mla_attn_decode(q_lat, d.q_pe, kv_rows, d.seq_start, d.seq_len, max_len, ws, o_lat)
    else:
        mla.mla_attn_decode_q8_0(q_lat, d.q_pe, q8[0], q8[1], d.seq_start, d.seq_len, max_len, ws, o_lat)
    return o_lat


@pytest.mark.parametrize("q8", [False, True])
def test_decode_skips_and_reports_bad_sequences(q8):
    lengths = [300, 500, 64, 200, 100]
    x = W.make_inputs("v3_decode_b32", n_head=16, lengths=lengths)
    d = Dev(x)
    n = int(sum(lengths))
    rng = np.random.default_rng(4)
    q_lat_np = W.normal_f16(rng, (len(lengths), 16, 512))
    q_lat = f16_dev(q_lat_np)
    rows = np.concatenate([x.c_kv, x.k_pe], axis=1)
    # the cache handed over ends 5 rows before the last sequence does (still
    # inside the allocation); sequence 1 claims more rows than max_len; sequence
    # 2 is empty
    n_rows = n - 5
    max_len = 400
    seq_len = x.seq_len.copy()
    seq_len[2] = 0
    d.seq_len = torch.from_numpy(seq_len).cuda()
    if q8:
        codes, scales = O.quantize_q8_0(rows)
        kv_q = torch.from_numpy(codes).cuda()[:n_rows]
        kv_d = torch.from_numpy(np.ascontiguousarray(scales[:n_rows].T)).cuda()
        o_lat = _decode_lat(d, q_lat, None, max_len, (kv_q, kv_d))
        ref_rows = O.dequantize_q8_0(codes, scales)
        tol = TOL_Q8
    else:
        o_lat = _decode_lat(d, q_lat, d.kv[:n_rows], max_len)
        ref_rows, tol = rows, TOL_BF16
    assert mla.mla_get_device_error() == MLA_ERR_INVALID_ARG
    got = o_lat.float().cpu().numpy()
    good = [0, 3]
    ref, _ = O.decode_latent(q_lat_np[good], x.q_pe[good], ref_rows[:, :512], ref_rows[:, 512:],
                             x.seq_start[good], x.seq_len[good], x.wl.scale)
    assert_tol(got[good], ref, tol, "valid sequences beside skipped ones")
    assert not got[[1, 2, 4]].any()                # skipped: left as they were (zeros)
    assert mla.mla_get_device_error() == 0


# ---------------------------------------------------------------------------
# Host buffers with overlapped copies (pipeline.HostOverlap)
# ---------------------------------------------------------------------------
def test_host_overlap_gives_the_serial_results():
    from mla_latent_kv_lat_gb300 import pipeline as P
    x = W.make_inputs("lite_t256", T=200, q_pos0=56, n_kv=256)
    d0 = Dev(x)
    ref = mla.mla_prefill(d0.q_nope, d0.q_pe, d0.wk_b, d0.wv_b, 56, kv=d0.kv).o.clone()
    d = {"q_nope": d0.q_nope, "q_pe": d0.q_pe, "wk_b": d0.wk_b, "wv_b": d0.wv_b, "kv": d0.kv}
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    bufs = P.prefill_buffers(200, 16, n_kv=256)

    def step(dv, out):
        P.mla_prefill(dv["q_nope"], dv["q_pe"], dv["wk_b"], dv["wv_b"], 56, kv=dv["kv"],
                      bufs=P.PrefillBuffers(bufs.q_lat, bufs.o_lat, out, None, bufs.workspace))
    dev = [{k: torch.zeros_like(v) for k, v in d.items()} for _ in range(2)]
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    run = P.HostOverlap(host, dev, outs, step)
    ms = run.run(5)
    assert ms > 0
    assert mla.mla_get_device_error() == 0
    for s in range(2):                            # both slots ran the step on the copied inputs
        assert torch.equal(run.host_out[s], ref.cpu())
