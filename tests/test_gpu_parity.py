"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on seeded inputs.

Tolerances are those of the stated target: max|d|/max|ref| <= 1e-2 and
mean|d|/mean|ref| <= 2e-3 with a bf16 cache, 3e-2 / 5e-3 with a q8_0 cache.
Small cases compare every output element; full-size workloads compare >= 512
sampled query rows (always the first and the last, and rows at tile edges).
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_lat_gb300 as mla
from mla_latent_kv_lat_gb300 import workloads as W
from oracle import mla_oracle as O
from tests.gpu_util import TOL_BF16, TOL_Q8, Dev, assert_tol, bf16_dev, dev_f32, f16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from mla_latent_kv_lat_gb300 import build
    build.build()
    mla.load_library()
    assert mla.mla_get_device_error() == 0


def _check_no_device_error():
    assert mla.mla_get_device_error() == 0


def run_prefill(d: Dev, q_pos0, q8=False, lse=False):
    x = d.x
    bufs = mla.pipeline.prefill_buffers(x.q_nope.shape[0], x.wl.n_head, with_lse=lse)
    if q8:
        mla.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, q_pos0, kv_q=d.kv_q, kv_d=d.kv_d, bufs=bufs)
    else:
        mla.mla_prefill(d.q_nope, d.q_pe, d.wk_b, d.wv_b, q_pos0, kv=d.kv, bufs=bufs)
    torch.cuda.synchronize()
    _check_no_device_error()
    return bufs


def run_decode(d: Dev, q8=False):
    x = d.x
    max_len = int(x.seq_len.max())
    kw = dict(kv_q=d.kv_q, kv_d=d.kv_d) if q8 else dict(kv=d.kv)
    bufs = mla.mla_decode(d.q_nope, d.q_pe, d.wk_b, d.wv_b, d.seq_start, d.seq_len, max_len, **kw)
    torch.cuda.synchronize()
    _check_no_device_error()
    return bufs


def sampled_rows(T, q_pos0, k=512, tile=128):
    edges = [0, T - 1]
    for t in range(0, T, max(1, T // 16)):
        edges += [t, t + 1, t + tile - 1]
    for t in range(T):
        if (q_pos0 + t) % tile in (0, tile - 1) and len(edges) < 64:
            edges.append(t)
    return W.sample_rows(T, k, seed=0, must=tuple(edges))


# ---------------------------------------------------------------------------
# Single steps on seeded inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,T", [(16, 1), (16, 77), (16, 256), (128, 200), (48, 130)])
def test_absorb_q_matches_oracle(H, T):
    x = W.make_inputs("v3_chunk8192_at32768", n_head=H, T=T, q_pos0=0, n_kv=T)
    q_nope, wk_b = bf16_dev(x.q_nope), bf16_dev(x.wk_b)
    q_lat = torch.empty(T, H, 512, dtype=torch.float16, device="cuda")
    mla.mla_absorb_q(q_nope, wk_b, q_lat)
    got = dev_f32(q_lat)
    ref = O.absorb_q(x.q_nope, x.wk_b)
    # one fp16 rounding (half an ulp = 2^-11 relative) of an fp32 sum of 128 exact products
    assert np.all(np.abs(got - ref) <= 2.0 ** -10 * np.abs(ref) + 1e-5 * np.sqrt(np.mean(ref ** 2)))
    _check_no_device_error()


@pytest.mark.parametrize("H,T", [(16, 1), (16, 77), (128, 200), (32, 64)])
def test_late_decompress_matches_oracle(H, T):
    rng = np.random.default_rng(5)
    o_lat = W.normal_f16(rng, (T, H, 512), 0.3)
    wv_b = W.normal_bf16(rng, (H, 512, 128), 1 / np.sqrt(512))
    o = torch.empty(T, H, 128, dtype=torch.float32, device="cuda")
    mla.mla_late_decompress(f16_dev(o_lat), bf16_dev(wv_b), o)
    got = o.cpu().numpy().astype(np.float64)
    ref = O.late_decompress(o_lat, wv_b)
    # fp32 accumulation of 512 bf16 x bf16 products (products exact in fp32)
    assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref)) + 1e-6
    _check_no_device_error()


@pytest.mark.parametrize("H,T,q_pos0,n_kv", [(16, 256, 0, 256), (16, 100, 37, 200), (128, 33, 300, 333),
                                            (16, 1, 0, 1), (64, 130, 0, 130)])
def test_prefill_latent_attention_matches_oracle(H, T, q_pos0, n_kv):
    x = W.make_inputs("lite_t256", n_head=H, T=T, q_pos0=q_pos0, n_kv=n_kv)
    rng = np.random.default_rng(3)
    q_lat = W.normal_f16(rng, (T, H, 512))
    d = Dev(x)
    o_lat = torch.empty(T, H, 512, dtype=torch.float16, device="cuda")
    lse = torch.empty(T, H, dtype=torch.float32, device="cuda")
    mla.mla_attn_prefill(f16_dev(q_lat), d.q_pe, d.kv, q_pos0, o_lat, lse)
    ref, ref_lse = O.attention_latent(q_lat, x.q_pe, x.c_kv, x.k_pe, x.q_pos(), x.wl.scale)
    assert_tol(dev_f32(o_lat), ref, TOL_BF16, "o_lat")
    # lse = log sum exp(s) moves by at most the largest score error.  Each score
    # is the sum of two fp16-rounded partial dot products (half an ulp: 2^-11
    # relative each), so the bound is 2^-11 * (|S_0| + |S_1|) * scale per key,
    # plus 2^-11 * 8 * ln 2 for the fp16 exponent argument (|arg| <= 8).
    half = 256
    s0 = np.abs(np.einsum("thc,jc->thj", q_lat[..., :half].astype(np.float64), x.c_kv[:, :half])
                + np.einsum("thr,jr->thj", x.q_pe.astype(np.float64), x.k_pe))
    s1 = np.abs(np.einsum("thc,jc->thj", q_lat[..., half:].astype(np.float64), x.c_kv[:, half:]))
    bound = 2.0 ** -11 * (s0 + s1).max() * x.wl.scale + 2.0 ** -11 * 8 * np.log(2) + 1e-5
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got_lse - ref_lse)) <= bound
    # and, independently of that kernel-derived bound, the normaliser exp(lse)
    # itself within the stated 1e-2 relative level of the oracle's
    assert np.max(np.abs(np.expm1(got_lse - ref_lse))) <= 1e-2
    _check_no_device_error()


# ---------------------------------------------------------------------------
# The whole path vs the un-absorbed definition
# ---------------------------------------------------------------------------
def test_prefill_chain_lite_t256_every_row():
    x = W.make_inputs("lite_t256")
    bufs = run_prefill(Dev(x), x.wl.q_pos0)
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_BF16, "lite_t256 o")


def test_prefill_chain_lite_t4096_every_row():
    x = W.make_inputs("lite_t4096")
    bufs = run_prefill(Dev(x), x.wl.q_pos0)
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_BF16, "lite_t4096 o")


def test_full_prefill_v3_chunk_sampled_rows():
    x = W.make_inputs("v3_chunk8192_at32768")
    bufs = run_prefill(Dev(x), x.wl.q_pos0)
    rows = sampled_rows(x.wl.T, x.wl.q_pos0)
    assert len(rows) >= 512
    ref, _ = O.attention_unabsorbed(x.q_nope[rows], x.q_pe[rows], x.c_kv, x.k_pe, x.wk_b, x.wv_b,
                                    x.q_pos()[rows], x.wl.scale)
    assert_tol(bufs.o.cpu().numpy()[rows], ref, TOL_BF16, "v3 chunk o")


def _decode_refs(x, c_kv, k_pe, n_heads_unabsorbed=4):
    """Absorbed-form oracle for every head (pinned to the definition by the
    associativity tests) plus the un-absorbed definition on sampled heads."""
    q_lat = O.absorb_q(x.q_nope, x.wk_b)
    o_lat, _ = O.decode_latent(q_lat, x.q_pe, c_kv, k_pe, x.seq_start, x.seq_len, x.wl.scale)
    ref = O.late_decompress(o_lat, x.wv_b)
    heads = list(W.sample_rows(x.wl.n_head, n_heads_unabsorbed, seed=1, must=(0, x.wl.n_head - 1)))
    ref_u = O.decode_unabsorbed(x.q_nope, x.q_pe, c_kv, k_pe, x.wk_b, x.wv_b, x.seq_start, x.seq_len,
                                x.wl.scale, heads=heads, seqs=[0, len(x.seq_len) - 1])
    return ref, heads, ref_u


def test_decode_chain_v3_b32_every_sequence():
    x = W.make_inputs("v3_decode_b32")
    bufs = run_decode(Dev(x))
    got = bufs.o.cpu().numpy()
    ref, heads, ref_u = _decode_refs(x, x.c_kv, x.k_pe, 2)
    assert_tol(got, ref, TOL_BF16, "decode o")
    assert_tol(got[[0, -1]][:, heads], ref_u, TOL_BF16, "decode o (un-absorbed heads)")


# Many short sequences (more than there are clusters): every cluster runs
# several pieces back to back, so the per-piece barrier phases (Q hand-over,
# output hand-over, row sums) turn over many times within one launch.
MANY_SHORT = [1 + (37 * i) % 300 for i in range(100)]


@pytest.mark.parametrize("lengths", [[1], [1, 2, 3], [2049, 4096, 17, 6000], [5000] * 3, MANY_SHORT])
def test_decode_chain_ragged_lengths(lengths):
    x = W.make_inputs("v3_decode_b32", n_head=32, lengths=lengths)
    bufs = run_decode(Dev(x))
    ref, heads, ref_u = _decode_refs(x, x.c_kv, x.k_pe)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_BF16, "decode o")


def test_decode_equals_last_prefill_row_on_gpu():
    x = W.make_inputs("lite_t256", T=300, n_kv=300, n_head=16)
    d = Dev(x)
    pre = run_prefill(d, 0)
    xd = W.Inputs(W.make_inputs("v3_decode_b32", n_head=16, lengths=[300]).wl, x.c_kv, x.k_pe,
                  x.q_nope[-1:], x.q_pe[-1:], x.wk_b, x.wv_b, np.array([300], np.int32), np.array([0], np.int64))
    dd = Dev(xd)
    dec = run_decode(dd)
    a, b = pre.o.cpu().numpy()[-1], dec.o.cpu().numpy()[0]
    assert_tol(b, a, (2e-3, 5e-4), "decode vs last prefill row")


# ---------------------------------------------------------------------------
# q8_0 cache
# ---------------------------------------------------------------------------
def test_quantize_q8_0_bit_exact():
    rng = np.random.default_rng(9)
    x = W.normal_bf16(rng, (1000, 576))
    x[3] = 0.0                                       # all-zero row: codes 0, scale 0
    x[5, :32] = np.float32(1e-30)                    # tiny block
    x[7, 64:96] *= 1000.0                            # large block
    x = W.to_bf16(x)[0]
    codes, scales = O.quantize_q8_0(x)
    kv = bf16_dev(x)
    kv_q = torch.empty(1000, 576, dtype=torch.int8, device="cuda")
    kv_d = torch.empty(18, 1024, dtype=torch.float16, device="cuda")
    mla.mla_quantize_q8_0(kv, kv_q, kv_d)
    np.testing.assert_array_equal(kv_q.cpu().numpy(), codes)
    np.testing.assert_array_equal(kv_d.cpu().numpy()[:, :1000].view(np.uint16), scales.T.view(np.uint16))
    _check_no_device_error()


def _q8(x: W.Inputs):
    codes, scales = O.quantize_q8_0(np.concatenate([x.c_kv, x.k_pe], axis=1))
    deq = O.dequantize_q8_0(codes, scales)
    return (codes, scales), deq[:, :512], deq[:, 512:]


def test_prefill_chain_q8_small_every_row():
    x = W.make_inputs("v3_q8_chunk8192_at90112", n_head=16, T=200, q_pos0=57, n_kv=300)
    q8, c_kv, k_pe = _q8(x)
    bufs = run_prefill(Dev(x, q8), x.wl.q_pos0, q8=True)
    ref, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, c_kv, k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_Q8, "q8 prefill o")


def test_full_prefill_q8_chunk_sampled_rows():
    x = W.make_inputs("v3_q8_chunk8192_at90112")
    q8, c_kv, k_pe = _q8(x)
    bufs = run_prefill(Dev(x, q8), x.wl.q_pos0, q8=True)
    rows = sampled_rows(x.wl.T, x.wl.q_pos0)
    ref, _ = O.attention_unabsorbed(x.q_nope[rows], x.q_pe[rows], c_kv, k_pe, x.wk_b, x.wv_b,
                                    x.q_pos()[rows], x.wl.scale)
    assert_tol(bufs.o.cpu().numpy()[rows], ref, TOL_Q8, "q8 chunk o")


def test_decode_chain_q8_b8_every_sequence():
    x = W.make_inputs("v3_q8_decode_b8")
    q8, c_kv, k_pe = _q8(x)
    bufs = run_decode(Dev(x, q8), q8=True)
    got = bufs.o.cpu().numpy()
    ref, heads, ref_u = _decode_refs(x, c_kv, k_pe, 2)
    assert_tol(got, ref, TOL_Q8, "q8 decode o")
    assert_tol(got[[0, -1]][:, heads], ref_u, TOL_Q8, "q8 decode o (un-absorbed heads)")


@pytest.mark.parametrize("lengths", [[1, 33, 2050], MANY_SHORT])
def test_decode_q8_small_ragged(lengths):
    x = W.make_inputs("v3_q8_decode_b8", n_head=16, lengths=lengths)
    q8, c_kv, k_pe = _q8(x)
    bufs = run_decode(Dev(x, q8), q8=True)
    ref, _, _ = _decode_refs(x, c_kv, k_pe)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_Q8, "q8 decode o")


# ---------------------------------------------------------------------------
# Invariants on the GPU
# ---------------------------------------------------------------------------
def test_prefill_is_deterministic_and_causal():
    x = W.make_inputs("lite_t256", T=200, q_pos0=100, n_kv=400)
    d = Dev(x)
    a = run_prefill(d, 100).o_lat.clone()
    b = run_prefill(d, 100).o_lat.clone()
    assert torch.equal(a, b)
    # rows past the last query's position are never read: garbage there changes nothing
    d.kv[300:] = float("nan")
    c = run_prefill(d, 100).o_lat.clone()
    assert torch.equal(a, c)


def test_wait_timeout_is_reported_and_cleared():
    assert mla.mla_get_device_error() == 0
    mla.mla_selftest_wait_timeout(1000)
    assert mla.mla_get_device_error() == -6          # MLA_ERR_TIMEOUT
    assert mla.mla_get_device_error() == 0           # read clears it
    x = W.make_inputs("lite_t256", T=16, n_kv=16)
    run_prefill(Dev(x), 0)                           # the context is still usable


def test_invalid_arguments_return_status():
    x = W.make_inputs("lite_t256", T=8, n_kv=8)
    d = Dev(x)
    o_lat = torch.empty(8, 16, 512, dtype=torch.float16, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_attn_prefill(f16_dev(np.zeros((8, 16, 512), np.float32)), d.q_pe, d.kv, 1, o_lat)
    assert e.value.status == -1                      # q_pos0 + T > n_kv
    with pytest.raises(mla.MLAError) as e:
        mla.mla_attn_prefill(f16_dev(np.zeros((8, 16, 512), np.float32)), d.q_pe, d.kv, 0, o_lat,
                             workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -4                      # prefill workspace too small
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.mla_attn_decode(o_lat[:1], d.q_pe[:1], d.kv, torch.zeros(1, dtype=torch.int64, device="cuda"),
                            torch.ones(1, dtype=torch.int32, device="cuda"), 8, ws, o_lat[:1])
    assert e.value.status == -4                      # workspace too small
    _check_no_device_error()


# ---------------------------------------------------------------------------
# The step before the path: mla_rope_append writes new tokens' cache rows
# ---------------------------------------------------------------------------
# The entry point takes freq_base / freq_scale as float (as ggml keeps them):
# the oracle turns by the same values (0.025 is not a float; its float is
# 1.5e-8 larger, which moves angles near 2000 rad by 3e-5).
FB, FS = float(np.float32(10000.0)), float(np.float32(0.025))


def _append_dev(a: W.AppendInputs):
    c = torch.from_numpy(W.to_bf16(a.c_kv)[1]).view(torch.bfloat16).cuda()
    k = torch.from_numpy(W.to_bf16(a.k_pe)[1]).view(torch.bfloat16).cuda()
    return c, k, torch.from_numpy(a.pos).cuda(), torch.from_numpy(a.slot).cuda()


def _caches(n_rows, ld_d):
    kv = torch.zeros(n_rows, 576, dtype=torch.bfloat16, device="cuda")
    kv_q = torch.zeros(n_rows, 576, dtype=torch.int8, device="cuda")
    kv_d = torch.zeros(18, ld_d, dtype=torch.float16, device="cuda")
    return kv, kv_q, kv_d


# 40001 tokens: more than one pass of the kernel's grid-stride loop over groups
# of four tokens (one pass covers 4 tokens x 8 warps x 8 blocks per SM), and
# not a multiple of four.
@pytest.mark.parametrize("n,n_rows", [(1, 4), (333, 1000), (4096, 98304), (40001, 98304)])
def test_rope_append_matches_oracle(n, n_rows):
    a = W.make_append_inputs(n, n_rows, seed=n)
    c, k, pos, slot = _append_dev(a)
    kv, kv_q, kv_d = _caches(n_rows, n_rows + 3)
    mla.mla_rope_append(c, k, pos, slot, kv=kv, kv_q=kv_q, kv_d=kv_d, freq_base=FB, freq_scale=FS)
    torch.cuda.synchronize()
    _check_no_device_error()
    got = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = W.to_bf16(O.cache_rows(a.c_kv, a.k_pe, a.pos, FB, FS).astype(np.float32))[1]
    rows = got[a.slot]
    # The latent part is copied: bit-exact.  The RoPE part: the device takes
    # the angle as an exact 0.64 fixed-point fraction of a turn (pos x frac(t_i)
    # modulo one turn), feeds its top 32 bits to sincospif (angle error
    # < 2^-23 rad from the truncation, plus sincospif's own few-ulp fp32 error),
    # rotates in fp32 and rounds once to bf16.  So the result is within half a
    # bf16 step (2^-8 relative) of the exact rotation, plus ~1e-6 of the pair's
    # magnitude from the fp32 sine, cosine and products (which matters only
    # where the two terms cancel).
    assert np.array_equal(rows[:, :512], ref[:, :512])
    exact = O.cache_rows(a.c_kv, a.k_pe, a.pos, FB, FS)[:, 512:]
    pair = np.repeat(np.maximum(np.abs(a.k_pe[:, 0::2]), np.abs(a.k_pe[:, 1::2])), 2, axis=1).astype(np.float64)
    err = np.abs(W.bf16_bits_to_f32(rows[:, 512:]).astype(np.float64) - exact)
    assert (err <= 2.0 ** -8 * np.abs(exact) + 1e-6 * pair).all()
    assert (rows[:, 512:] != ref[:, 512:]).mean() < 1e-2
    # rows not written stay untouched
    untouched = np.setdiff1d(np.arange(n_rows), a.slot)
    assert not got[untouched].any()
    # the q8_0 rows: the oracle's quantisation of the device's own bf16 rows, bit-exact
    codes, scales = O.quantize_q8_0(W.bf16_bits_to_f32(rows))
    assert np.array_equal(kv_q.cpu().numpy()[a.slot], codes)
    got_d = kv_d.cpu().numpy()
    assert np.array_equal(got_d[:, a.slot].T.view(np.uint16), scales.view(np.uint16))
    assert not got_d[:, n_rows:].view(np.uint16).any()
    # one cache at a time writes the same rows
    kv2, kq2, kd2 = _caches(n_rows, n_rows + 3)
    mla.mla_rope_append(c, k, pos, slot, kv=kv2)
    mla.mla_rope_append(c, k, pos, slot, kv_q=kq2, kv_d=kd2)
    torch.cuda.synchronize()
    assert torch.equal(kv2.view(torch.int16), kv.view(torch.int16))
    assert torch.equal(kq2, kv_q) and torch.equal(kd2.view(torch.int16), kv_d.view(torch.int16))


def test_rope_append_then_decode_reads_the_rows():
    # a sequence whose rows were all written by mla_rope_append (positions
    # 0..L-1, the RoPE part rotated by position) decodes as the oracle does
    # on those rows
    L, H = 700, 32
    a = W.make_append_inputs(L, L, seed=11)
    a.pos[:] = np.arange(L, dtype=np.int32)
    a.slot[:] = np.arange(L, dtype=np.int64)
    c, k, pos, slot = _append_dev(a)
    kv, kv_q, kv_d = _caches(L, L)
    mla.mla_rope_append(c, k, pos, slot, kv=kv, kv_q=kv_q, kv_d=kv_d)
    torch.cuda.synchronize()
    _check_no_device_error()
    x = W.make_inputs("v3_decode_b32", n_head=H, lengths=[L])
    rows = W.bf16_bits_to_f32(kv.view(torch.int16).cpu().numpy().view(np.uint16))
    x = W.Inputs(x.wl, rows[:, :512], rows[:, 512:], x.q_nope, x.q_pe, x.wk_b, x.wv_b, x.seq_len, x.seq_start)
    d = Dev(x)
    d.kv = kv                                   # decode reads the cache the append wrote
    bufs = run_decode(d)
    ref, _, _ = _decode_refs(x, x.c_kv, x.k_pe)
    assert_tol(bufs.o.cpu().numpy(), ref, TOL_BF16, "decode o on appended rows")


@pytest.mark.parametrize("bad", ["slot", "pos"])
def test_rope_append_out_of_range_slot_is_skipped_and_reported(bad):
    # token 3 is bad (slot one past the end, or a negative position); tokens
    # 0..2 share its group of four tokens in the kernel's RoPE pass, so their
    # RoPE columns and q8_0 rows are where a masking mistake would show
    a = W.make_append_inputs(8, 16, seed=3)
    if bad == "slot":
        a.slot[3] = 16
    else:
        a.pos[3] = -5
    c, k, pos, slot = _append_dev(a)
    kv, kv_q, kv_d = _caches(16, 16)
    mla.mla_rope_append(c, k, pos, slot, kv=kv, kv_q=kv_q, kv_d=kv_d, freq_base=FB, freq_scale=FS)
    assert mla.mla_get_device_error() == -1     # MLA_ERR_INVALID_ARG, read and cleared
    got = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    ok = [j for j in range(8) if j != 3]
    exact = O.cache_rows(a.c_kv[ok], a.k_pe[ok], a.pos[ok], FB, FS)
    ref = W.to_bf16(exact.astype(np.float32))[1]
    rows = got[a.slot[ok]]
    assert np.array_equal(rows[:, :512], ref[:, :512])
    pair = np.repeat(np.maximum(np.abs(a.k_pe[ok, 0::2]), np.abs(a.k_pe[ok, 1::2])), 2, axis=1).astype(np.float64)
    err = np.abs(W.bf16_bits_to_f32(rows[:, 512:]).astype(np.float64) - exact[:, 512:])
    assert (err <= 2.0 ** -8 * np.abs(exact[:, 512:]) + 1e-6 * pair).all()
    codes, scales = O.quantize_q8_0(W.bf16_bits_to_f32(rows))
    assert np.array_equal(kv_q.cpu().numpy()[a.slot[ok]], codes)
    assert np.array_equal(kv_d.cpu().numpy()[:, a.slot[ok]].T.view(np.uint16), scales.view(np.uint16))
    # every other row, the bad token's neighbours in the cache included, is untouched
    untouched = np.setdiff1d(np.arange(16), a.slot[ok])
    assert not got[untouched].any()
    assert not kv_q.cpu().numpy()[untouched].any()
    assert not kv_d.cpu().numpy()[:, untouched].view(np.uint16).any()
    assert mla.mla_get_device_error() == 0
