"""CUDA graph capture of the path's steps.

Every launch of the library takes its stream as an argument and allocates
nothing, so a step (absorb -> attention -> late decompression, or a decode
step with its split-KV combine, a programmatic dependent launch) can be
captured once and replayed: the replay skips the host work of each call
(argument checks, tensor-map encoding, launches).  A captured step replayed
on new inputs copied into its buffers must give the bits of the same call
made eagerly on those inputs, and match the oracle.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_lat_gb300 as mla
from mla_latent_kv_lat_gb300 import pipeline as P
from mla_latent_kv_lat_gb300 import workloads as W
from oracle import mla_oracle as O
from tests.gpu_util import TOL_BF16, TOL_Q8, Dev, assert_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from mla_latent_kv_lat_gb300 import build
    build.build()
    mla.load_library()
    assert mla.mla_get_device_error() == 0


def _capture(step):
    """Run `step` once eagerly (first-call lookups happen outside capture),
    then capture it on a side stream."""
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _refill(dst: Dev, src: Dev, names):
    for n in names:
        getattr(dst, n).copy_(getattr(src, n))


@pytest.mark.parametrize("q8", [False, True])
def test_decode_step_replays_eager_bits(q8):
    lengths = [700, 64, 1500, 333, 1]
    H, max_len = 32, 2048
    mk = lambda seed: W.make_inputs("v3_decode_b32", seed, n_head=H, lengths=lengths)
    quant = (lambda x: O.quantize_q8_0(np.concatenate([x.c_kv, x.k_pe], axis=1))) if q8 else (lambda x: None)
    x0 = mk(0)
    d = Dev(x0, quant(x0))
    bufs = P.decode_buffers(len(lengths), H, max_len)
    cache = dict(kv_q=d.kv_q, kv_d=d.kv_d) if q8 else dict(kv=d.kv)

    def step():
        P.mla_decode(d.q_nope, d.q_pe, d.wk_b, d.wv_b, d.seq_start, d.seq_len, max_len, bufs=bufs, **cache)

    g = _capture(step)
    names = ["q_nope", "q_pe", "wk_b", "wv_b"] + (["kv_q", "kv_d"] if q8 else ["kv"])
    for seed in (1, 2):
        x = mk(seed)
        new = Dev(x, quant(x))
        _refill(d, new, names)
        g.replay()
        torch.cuda.synchronize()
        got = bufs.o.clone()
        eager_cache = dict(kv_q=new.kv_q, kv_d=new.kv_d) if q8 else dict(kv=new.kv)
        eager = P.mla_decode(new.q_nope, new.q_pe, new.wk_b, new.wv_b, new.seq_start, new.seq_len, max_len,
                             **eager_cache)
        torch.cuda.synchronize()
        assert torch.equal(got, eager.o)
        assert mla.mla_get_device_error() == 0
    # the last replay against the oracle (un-absorbed heads, the decoded rows of each sequence)
    rows = np.concatenate([x.c_kv, x.k_pe], axis=1)
    if q8:
        rows = O.dequantize_q8_0(*O.quantize_q8_0(rows))
    ref = O.decode_unabsorbed(x.q_nope, x.q_pe, rows[:, :512], rows[:, 512:], x.wk_b, x.wv_b, x.seq_start,
                              x.seq_len, x.wl.scale)
    assert_tol(got.cpu().numpy().astype(np.float64), ref, TOL_Q8 if q8 else TOL_BF16, "decode graph replay o")


def test_static_decode_replays_eager_bits():
    lengths = [900, 65, 4096]
    H, max_len = 64, 4096
    x0 = W.make_inputs("v3_decode_b32", 0, n_head=H, lengths=lengths)
    d = Dev(x0)
    rng = np.random.default_rng(5)
    q_lat = torch.from_numpy(W.to_f16(W.normal_f16(rng, (len(lengths), H, 512)))[1]).view(torch.float16).cuda()
    o_lat = torch.empty(len(lengths), H, 512, dtype=torch.float16, device="cuda")
    g = _capture(lambda: mla.mla_attn_decode_static(q_lat, d.q_pe, d.kv, d.seq_start, d.seq_len, max_len, o_lat))
    for seed in (6, 7):
        q_new = torch.from_numpy(W.to_f16(W.normal_f16(np.random.default_rng(seed), q_lat.shape))[1])
        q_lat.copy_(q_new.view(torch.float16).cuda())
        g.replay()
        torch.cuda.synchronize()
        got = o_lat.clone()
        eager = torch.empty_like(o_lat)
        mla.mla_attn_decode_static(q_lat, d.q_pe, d.kv, d.seq_start, d.seq_len, max_len, eager)
        torch.cuda.synchronize()
        assert torch.equal(got, eager)
    assert mla.mla_get_device_error() == 0


def test_prefill_step_replays_eager_bits():
    mk = lambda seed: W.make_inputs("lite_t256", seed, T=200, q_pos0=56, n_kv=256)
    x0 = mk(0)
    d = Dev(x0)
    bufs = P.prefill_buffers(200, 16, n_kv=256)

    def step():
        P.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, 56, kv=d.kv, bufs=bufs)

    g = _capture(step)
    for seed in (1, 2):
        x = mk(seed)
        new = Dev(x)
        _refill(d, new, ["q_nope", "q_pe", "wk_b", "wv_b", "kv"])
        g.replay()
        torch.cuda.synchronize()
        got = bufs.o.clone()
        eager = P.mla_prefill(new.q_nope, new.q_pe, new.wk_b, new.wv_b, 56, kv=new.kv)
        torch.cuda.synchronize()
        assert torch.equal(got, eager.o)
    assert mla.mla_get_device_error() == 0
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(got.cpu().numpy().astype(np.float64), ref, TOL_BF16, "prefill graph replay o")
