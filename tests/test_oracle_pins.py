"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: a brute-force scalar implementation on tiny inputs, closed forms and
special cases of softmax attention, the associativity identity the method
rests on ("MLA matrix absorption in ik_llama.cpp", sec. 2), the causal rule,
the pages' own layouts and einsums (sec. 4-5 and PR #394 sec. 3.2), and the
numbers the pages print (tests/golden/page_accounting.json).
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O
from mla_latent_kv_lat_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_case(seed, H=2, L=8, R=4, Dn=4, Dv=4, T=5, N=9, q_pos0=None):
    rng = np.random.default_rng(seed)
    if q_pos0 is None:
        q_pos0 = N - T
    return dict(
        q_nope=rng.standard_normal((T, H, Dn)), q_pe=rng.standard_normal((T, H, R)),
        c_kv=rng.standard_normal((N, L)), k_pe=rng.standard_normal((N, R)),
        wk_b=rng.standard_normal((H, Dn, L)) / math.sqrt(Dn),
        wv_b=rng.standard_normal((H, L, Dv)) / math.sqrt(L),
        q_pos=q_pos0 + np.arange(T), scale=1.0 / math.sqrt(Dn + R))


def brute_force(q_nope, q_pe, c_kv, k_pe, wk_b, wv_b, q_pos, scale):
    """Scalar loops, no numpy arithmetic: decompress, 192-d dot, softmax, weighted sum."""
    T, H, Dn = q_nope.shape
    L = c_kv.shape[1]
    R = k_pe.shape[1]
    Dv = wv_b.shape[2]
    out = np.zeros((T, H, Dv))
    for t in range(T):
        for h in range(H):
            keys = range(int(q_pos[t]) + 1)
            scores = []
            for j in keys:
                s = 0.0
                for d in range(Dn):
                    k = 0.0
                    for c in range(L):
                        k += float(wk_b[h, d, c]) * float(c_kv[j, c])
                    s += float(q_nope[t, h, d]) * k
                for r in range(R):
                    s += float(q_pe[t, h, r]) * float(k_pe[j, r])
                scores.append(scale * s)
            mx = max(scores)
            w = [math.exp(x - mx) for x in scores]
            z = sum(w)
            for e in range(Dv):
                acc = 0.0
                for j, wj in zip(keys, w):
                    v = 0.0
                    for c in range(L):
                        v += float(wv_b[h, c, e]) * float(c_kv[j, c])
                    acc += wj / z * v
                out[t, h, e] = acc
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_unabsorbed_matches_brute_force(seed):
    cs = tiny_case(seed)
    o, _ = O.attention_unabsorbed(**cs)
    ref = brute_force(**cs)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 3])
def test_absorbed_chain_matches_brute_force(seed):
    cs = tiny_case(seed, q_pos0=2)
    o, _, _ = O.attention_absorbed(**cs)
    np.testing.assert_allclose(o, brute_force(**cs), rtol=0, atol=1e-12)


def test_associativity_on_lite_shape():
    """sec. 2: un-absorbed and absorbed are the same function (fp64, DeepSeek-Lite shape)."""
    x = W.make_inputs("lite_t256", T=64, n_kv=64)
    args = (x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    o_u, lse_u = O.attention_unabsorbed(*args)
    o_a, _, lse_a = O.attention_absorbed(*args)
    assert np.max(np.abs(o_u - o_a)) <= 1e-12 * np.max(np.abs(o_u))
    np.testing.assert_allclose(lse_u, lse_a, rtol=1e-13, atol=0)


def test_first_position_sees_only_row_zero():
    """A query at position 0 attends row 0 alone, so o[h] = W^UV_h c_0 for any query."""
    cs = tiny_case(4, T=1, q_pos0=0)
    o, lse = O.attention_unabsorbed(**cs)
    for h in range(2):
        v0 = np.array([sum(cs["wv_b"][h, c, e] * cs["c_kv"][0, c] for c in range(8)) for e in range(4)])
        np.testing.assert_allclose(o[0, h], v0, atol=1e-13)
        s0 = cs["scale"] * (sum(cs["q_pe"][0, h, r] * cs["k_pe"][0, r] for r in range(4))
                            + sum(cs["q_nope"][0, h, d] * sum(cs["wk_b"][h, d, c] * cs["c_kv"][0, c]
                                                              for c in range(8)) for d in range(4)))
        assert abs(lse[0, h] - s0) < 1e-12


def test_identical_rows_make_output_independent_of_query():
    cs = tiny_case(5)
    cs["c_kv"][:] = cs["c_kv"][0]
    cs["k_pe"][:] = cs["k_pe"][0]
    o1, _ = O.attention_unabsorbed(**cs)
    cs2 = dict(cs, q_nope=cs["q_nope"] * -3.0 + 1.0, q_pe=cs["q_pe"] * 2.0)
    o2, _ = O.attention_unabsorbed(**cs2)
    np.testing.assert_allclose(o1, o2, atol=1e-13)


def test_zero_query_gives_mean_of_visible_rows():
    cs = tiny_case(6, q_pos0=0)
    cs["q_nope"][:] = 0.0
    cs["q_pe"][:] = 0.0
    o, lat, lse = O.attention_absorbed(**cs)
    for t in range(5):
        n = t + 1
        np.testing.assert_allclose(lat[t, 0], cs["c_kv"][:n].mean(axis=0), atol=1e-13)
        np.testing.assert_allclose(lse[t], math.log(n), atol=1e-13)


def test_constant_rope_score_shift_changes_nothing():
    """Equal k_pe rows add q_pe.u to every score of a row: p unchanged, lse shifted."""
    cs = tiny_case(7)
    u = cs["k_pe"][0].copy()
    cs["k_pe"][:] = u
    o1, lse1 = O.attention_unabsorbed(**cs)
    o0, lse0 = O.attention_unabsorbed(**dict(cs, q_pe=np.zeros_like(cs["q_pe"])))
    np.testing.assert_allclose(o1, o0, atol=1e-13)
    shift = cs["scale"] * np.einsum("thr,r->th", cs["q_pe"], u)
    np.testing.assert_allclose(lse1 - lse0, shift, atol=1e-12)


def test_causal_rows_beyond_position_are_ignored_bitwise():
    cs = tiny_case(8, T=4, N=12, q_pos0=3)
    o1, l1 = O.attention_unabsorbed(**cs)
    a1, b1 = O.attention_latent(O.absorb_q(cs["q_nope"], cs["wk_b"]), cs["q_pe"], cs["c_kv"], cs["k_pe"],
                                cs["q_pos"], cs["scale"])
    for t in range(4):
        # garbage in every row after query t's position: row t's result must not move
        g = dict(cs)
        g["c_kv"] = cs["c_kv"].copy()
        g["k_pe"] = cs["k_pe"].copy()
        g["c_kv"][cs["q_pos"][t] + 1:] = 1e6
        g["k_pe"][cs["q_pos"][t] + 1:] = -1e6
        o2, l2 = O.attention_unabsorbed(**g)
        assert np.array_equal(o1[t], o2[t]) and np.array_equal(l1[t], l2[t])
        a2, b2 = O.attention_latent(O.absorb_q(g["q_nope"], g["wk_b"]), g["q_pe"], g["c_kv"], g["k_pe"],
                                    g["q_pos"], g["scale"])
        assert np.array_equal(a1[t], a2[t]) and np.array_equal(b1[t], b2[t])


def test_decode_equals_last_prefill_row():
    x = W.make_inputs("lite_t256", T=32, n_kv=32)
    o_p, _ = O.attention_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    o_d = O.decode_unabsorbed(x.q_nope[-1:], x.q_pe[-1:], x.c_kv, x.k_pe, x.wk_b, x.wv_b,
                              np.array([0]), np.array([32]), x.wl.scale)
    np.testing.assert_allclose(o_d[0], o_p[-1], atol=1e-14)
    q_lat = O.absorb_q(x.q_nope[-1:], x.wk_b)
    lat_d, _ = O.decode_latent(q_lat, x.q_pe[-1:], x.c_kv, x.k_pe, np.array([0]), np.array([32]), x.wl.scale)
    _, lat_p, _ = O.attention_absorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.q_pos(), x.wl.scale)
    np.testing.assert_allclose(lat_d[0], lat_p[-1], atol=1e-13)


def test_decode_sequences_use_their_own_rows():
    """Each sequence's query sits at position len-1 over its own packed rows."""
    lens = [3, 7, 5]
    starts = np.array([0, 3, 10])
    cs = tiny_case(11, T=3, N=15)
    o = O.decode_unabsorbed(cs["q_nope"], cs["q_pe"], cs["c_kv"], cs["k_pe"], cs["wk_b"], cs["wv_b"],
                            starts, np.array(lens), cs["scale"])
    for b in range(3):
        s0, n = int(starts[b]), lens[b]
        ref = brute_force(cs["q_nope"][b:b + 1], cs["q_pe"][b:b + 1], cs["c_kv"][s0:s0 + n],
                          cs["k_pe"][s0:s0 + n], cs["wk_b"], cs["wv_b"], [n - 1], cs["scale"])
        np.testing.assert_allclose(o[b], ref[0], atol=1e-12)


def test_pages_layouts_and_einsums_agree():
    """sec. 4-5 einsums with the pages' weight layouts give the oracle's o.

    PR #394 sec. 3.2: mainline wk_b has ggml shape {128, 512, H}, i.e. row-major
    [H][512][128]; the sec. 4 einsum 'bhqc,hdc->bhqd' stores W_UV as [h][d][c].
    Both are transposes of the boundary layouts wk_b[H,128,512], wv_b[H,512,128].
    """
    cs = tiny_case(9, q_pos0=4)
    wk_ggml = np.ascontiguousarray(cs["wk_b"].transpose(0, 2, 1))    # [H][L][Dn]
    W_UV = np.ascontiguousarray(cs["wv_b"].transpose(0, 2, 1))       # [h][d][c]
    q = cs["q_nope"].transpose(1, 0, 2)[None]                        # b h q d
    q_lat = np.einsum("bhqd,hcd->bhqc", q, wk_ggml)                  # ggml_mul_mat(wk_b, q_nope)
    kv = cs["c_kv"][None]                                            # b l c
    s = (np.einsum("bhqr,blr->bhql", cs["q_pe"].transpose(1, 0, 2)[None], cs["k_pe"][None])
         + np.einsum("bhqc,blc->bhql", q_lat, kv)) * cs["scale"]
    mask = np.arange(kv.shape[1])[None, :] <= cs["q_pos"][:, None]
    s = np.where(mask[None, None], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    out = np.einsum("bhql,blc->bhqc", p, kv)
    out = np.einsum("bhqc,hdc->bhqd", out, W_UV)[0].transpose(1, 0, 2)
    o, _ = O.attention_unabsorbed(**cs)
    np.testing.assert_allclose(o, out, atol=1e-12)


def test_page_accounting_numbers():
    g = json.load(open(os.path.join(GOLDEN, "page_accounting.json")))
    items = {it["name"]: it for it in g["items"]}
    H = g["n_head_v3"]
    lat = O.latent_row_bytes(2)
    dec = O.decompressed_token_bytes(H, 2)
    assert lat == 1152 and round(lat / 1000, 2) == items["latent_cache_kb_per_token"]["value"]
    assert dec == 81920 and round(dec / 1000, 2) == items["decompressed_cache_kb_per_token"]["value"]
    f_dec = O.flops_per_pair_decompressed(H)
    f_lat = O.flops_per_token_decompress(H) + f_dec
    f_abs = O.flops_per_pair_absorbed(H)
    assert (f_dec, f_lat, f_abs) == (81920, 33636352, 278528)
    assert round(f_dec / 1e6, 2) == items["mflop_per_pair_decompressed"]["value"]
    assert round(f_lat / 1e6, 2) == items["mflop_per_token_latent_no_absorption"]["value"]
    assert round(f_abs / 1e6, 2) == items["mflop_per_pair_absorbed"]["value"]
    assert round(dec / lat) == items["cache_ratio"]["value"]
    assert round(f_lat / f_abs, -1) == items["flop_ratio"]["value"]
    assert round(100 * (1 - lat / dec), 1) == items["compression_percent"]["value"]
    it = items["q8_0_cache_mib"]
    assert O.q8_0_row_bytes() == 612
    mib = O.q8_0_row_bytes() * it["n_ctx"] * it["n_layer_reading"] / 2 ** 20
    assert mib == 3499.875 and round(mib + 1e-9, 2) == it["value"]
    assert H * (O.KV_LORA_RANK + O.QK_ROPE) == items["attn_q_b_expected_cols"]["value"]
    assert H * (O.QK_NOPE + O.QK_ROPE) == items["attn_q_b_got_cols"]["value"]
    assert O.KV_LORA_RANK + O.QK_ROPE == items["key_length"]["value"]
    assert O.KV_LORA_RANK == items["value_length"]["value"]
    assert O.QK_NOPE + O.QK_ROPE == items["key_length_mla"]["value"]
    assert O.V_HEAD == items["value_length_mla"]["value"]


def test_causal_pair_count():
    for T, p0 in [(1, 0), (5, 0), (5, 3), (256, 0), (8192, 32768)]:
        assert O.causal_pairs(T, p0) == sum(p0 + t + 1 for t in range(T))


# ---------------------------------------------------------------------------
# q8_0 (sec. 8.1; block size from the q8_0 cache size in discussion #586)
# ---------------------------------------------------------------------------
def test_q8_0_exact_codes_on_power_of_two_scale():
    """amax = 31.75 gives d = 0.25 exactly, so every x = 0.25 k maps back to k."""
    k = np.arange(-16, 16, dtype=np.int64) * 7 % 255 - 127
    k[0] = 127
    x = np.tile((0.25 * k).astype(np.float32), 18)[None, :]
    codes, d = O.quantize_q8_0(x)
    assert codes.dtype == np.int8 and d.dtype == np.float16 and d.shape == (1, 18)
    assert np.all(d == np.float16(0.25))
    np.testing.assert_array_equal(codes[0], np.tile(k, 18))
    np.testing.assert_array_equal(O.dequantize_q8_0(codes, d), x.astype(np.float64))


def test_q8_0_rounds_half_away_from_zero_and_zero_block():
    blk = np.zeros(32, np.float32)
    blk[0] = 31.75      # d = 0.25
    blk[1] = 0.625      # 2.5  -> 3
    blk[2] = -0.625     # -2.5 -> -3
    blk[3] = 0.375      # 1.5  -> 2
    blk[4] = 0.12       # 0.48 -> 0
    x = np.concatenate([blk, np.zeros(32 * 17, np.float32)])[None]
    codes, d = O.quantize_q8_0(x)
    assert list(codes[0, :5]) == [127, 3, -3, 2, 0]
    assert np.all(codes[0, 32:] == 0) and np.all(d[0, 1:] == 0)


def test_q8_0_error_bound_and_code_range():
    x = W.make_inputs("v3_q8_decode_b8", n_head=1, lengths=[64]).c_kv
    x = np.concatenate([x, x[:, :64]], axis=1)[:, :576]
    codes, d = O.quantize_q8_0(x)
    assert codes.min() >= -127 and codes.max() <= 127
    assert np.all(np.abs(codes.reshape(64, 18, 32)).max(axis=2) == 127)
    deq = O.dequantize_q8_0(codes, d).reshape(64, 18, 32)
    d32 = (np.abs(x.reshape(64, 18, 32)).max(axis=2) / np.float32(127)).astype(np.float64)
    bound = d32 / 2 + 127 * np.abs(d.astype(np.float64) - d32) + 1e-12
    assert np.all(np.abs(deq - x.reshape(64, 18, 32)).max(axis=2) <= bound)


# ---------------------------------------------------------------------------
# RoPE and the cache rows of new tokens ("llama.cpp KV Cache 与注意力机制"
# sec. 2.3; freq_base / freq_scale from the context log of "ik_llama.cpp
# discussion #586 slow KV cache rm")
# ---------------------------------------------------------------------------
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(5).standard_normal((7, 64))
    assert np.array_equal(O.rope_rotate(x, np.zeros(7), 10000.0, 0.025), x)


def test_rope_quarter_turn_of_pair_zero_closed_form():
    # pair 0 turns by pos * freq_scale (freq_base^0 = 1): at a quarter turn,
    # e_0 -> e_1 and e_1 -> -e_0, every other dimension untouched (pairing
    # (2i, 2i+1): a split-half pairing would move e_0 to e_32).
    pos = (math.pi / 2) / 0.025
    e0, e1 = np.zeros(64), np.zeros(64)
    e0[0], e1[1] = 1.0, 1.0
    r0 = O.rope_rotate(e0, pos, 10000.0, 0.025)
    r1 = O.rope_rotate(e1, pos, 10000.0, 0.025)
    assert abs(r0[1] - 1.0) < 1e-12 and np.abs(np.delete(r0, 1)).max() < 1e-12
    assert abs(r1[0] + 1.0) < 1e-12 and np.abs(np.delete(r1, 0)).max() < 1e-12


def test_rope_frequency_of_each_pair_closed_form():
    # pair i turns by pos * s * b^(-2i/64): read the angle back from e_(2i).
    b, s, pos = 10000.0, 0.025, 12345.0
    for i in range(32):
        e = np.zeros(64)
        e[2 * i] = 1.0
        r = O.rope_rotate(e, pos, b, s)
        theta = pos * s * b ** (-2.0 * i / 64)
        assert abs(r[2 * i] - math.cos(theta)) < 1e-9 and abs(r[2 * i + 1] - math.sin(theta)) < 1e-9


def test_rope_preserves_pair_norms_and_scale_acts_on_position():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 64))
    pos = rng.integers(0, 100000, 5).astype(np.float64)
    r = O.rope_rotate(x, pos, 10000.0, 0.025)
    n = lambda v: v[:, 0::2] ** 2 + v[:, 1::2] ** 2
    assert np.abs(n(r) - n(x)).max() < 1e-9
    assert np.abs(r - O.rope_rotate(x, pos * 0.025, 10000.0, 1.0)).max() < 1e-9


def test_rope_scores_depend_on_relative_position_only():
    # <R(m) q, R(n) k> = <R(m - n) q, k>: the property RoPE exists for.
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in [(10, 3), (5000, 4990), (98303, 17)]:
        lhs = O.rope_rotate(q, m, 10000.0, 0.025) @ O.rope_rotate(k, n, 10000.0, 0.025)
        rhs = O.rope_rotate(q, m - n, 10000.0, 0.025) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_cache_rows_keep_the_latent_part_and_rotate_the_rope_part():
    rng = np.random.default_rng(8)
    c, kp = rng.standard_normal((3, 512)), rng.standard_normal((3, 64))
    pos = np.array([0, 7, 90000])
    rows = O.cache_rows(c, kp, pos, 10000.0, 0.025)
    assert rows.shape == (3, 576)
    assert np.array_equal(rows[:, :512], c)
    assert np.array_equal(rows[0, 512:], kp[0])
    assert np.array_equal(rows[1:, 512:], O.rope_rotate(kp[1:], pos[1:], 10000.0, 0.025))


# ---------------------------------------------------------------------------
# The step after the path: the output projection (method page sec. 4, the
# einsum 'hdD,bhqd->bqD'; sec. 6 on folding W_O into W_UV)
# ---------------------------------------------------------------------------
def test_output_projection_matches_brute_force_loops():
    rng = np.random.default_rng(12)
    T, H, d, D = 3, 2, 4, 5
    o, w = rng.standard_normal((T, H, d)), rng.standard_normal((H, d, D))
    ref = np.zeros((T, D))
    for t in range(T):
        for n in range(D):
            ref[t, n] = sum(w[h, k, n] * o[t, h, k] for h in range(H) for k in range(d))
    np.testing.assert_allclose(O.output_projection(o, w), ref, atol=1e-12)


def test_output_projection_is_the_pages_einsum_and_folds_into_wv_b():
    # the page's own einsum on its [b, h, q, d] layout gives the same u; folding
    # W_O into W_UV per head (sec. 6) gives the same u from o_lat (associativity)
    rng = np.random.default_rng(13)
    T, H, L, d, D = 4, 3, 16, 8, 6
    o_lat, wv, wo = rng.standard_normal((T, H, L)), rng.standard_normal((H, L, d)), rng.standard_normal((H, d, D))
    o = O.late_decompress(o_lat, wv)
    u = O.output_projection(o, wo)
    page = np.einsum("hdD,bhqd->bqD", wo, o.transpose(1, 0, 2)[None])[0]
    np.testing.assert_allclose(u, page, atol=1e-12)
    folded = np.einsum("thc,hcD->tD", o_lat, O.projected_weights(wv, wo))
    np.testing.assert_allclose(u, folded, atol=1e-10)
    # one head's weights zero: that head drops out of the sum
    wo0 = wo.copy()
    wo0[1] = 0
    np.testing.assert_allclose(O.output_projection(o, wo0),
                               O.output_projection(o[:, [0, 2]], wo[[0, 2]]), atol=1e-12)


def test_rope_constants_are_the_pages_printed_values():
    # the cache-append defaults (binding and bench) are the printed freq_base /
    # freq_scale of the DeepSeek-V3 run, over the printed n_rot = 64 dims
    import inspect

    from mla_latent_kv_lat_gb300 import binding
    g = json.load(open(os.path.join(GOLDEN, "page_accounting.json")))
    items = {it["name"]: it for it in g["items"]}
    sig = inspect.signature(binding.mla_rope_append).parameters
    assert sig["freq_base"].default == items["rope_freq_base"]["value"]
    assert sig["freq_scale"].default == items["rope_freq_scale"]["value"]
    assert O.QK_ROPE == items["rope_n_rot"]["value"]
