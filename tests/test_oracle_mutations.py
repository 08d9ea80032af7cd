"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
of tests/test_oracle_pins.py notice each one."""
import math

import numpy as np
import pytest

from oracle import mla_oracle as O
from tests.test_oracle_pins import brute_force, tiny_case


def _mismatch(o, ref):
    return not np.allclose(o, ref, rtol=0, atol=1e-12)


def test_dropped_rope_term_is_caught():
    cs = tiny_case(0)
    ref = brute_force(**cs)
    o, _ = O.attention_unabsorbed(**dict(cs, k_pe=np.zeros_like(cs["k_pe"])))
    assert _mismatch(o, ref)


def test_off_by_one_causal_rule_is_caught():
    cs = tiny_case(1)
    ref = brute_force(**cs)
    o, _ = O.attention_unabsorbed(**dict(cs, q_pos=cs["q_pos"] - 1))
    assert _mismatch(o, ref)


def test_wrong_scale_is_caught():
    cs = tiny_case(2)
    ref = brute_force(**cs)
    o, _ = O.attention_unabsorbed(**dict(cs, scale=1.0 / math.sqrt(4)))
    assert _mismatch(o, ref)


@pytest.mark.parametrize("which", ["transpose_wk", "swap_kv", "sign_wv"])
def test_decompression_mistakes_are_caught(monkeypatch, which):
    cs = tiny_case(3, Dn=8, Dv=8, L=8)          # square per-head blocks so a transpose still runs
    ref = brute_force(**cs)
    good = O.decompress_head

    def bad(c_kv, wk, wv):
        if which == "transpose_wk":
            return good(c_kv, np.asarray(wk).T, wv)
        k, v = good(c_kv, wk, wv)
        return (v, k) if which == "swap_kv" else (k, -v)

    monkeypatch.setattr(O, "decompress_head", bad)
    o, _ = O.attention_unabsorbed(**cs)
    assert _mismatch(o, ref)


def test_transposed_absorption_is_caught():
    cs = tiny_case(4, Dn=8, L=8)
    ref = brute_force(**cs)
    wk_t = np.ascontiguousarray(cs["wk_b"].transpose(0, 2, 1))
    o, _, _ = O.attention_absorbed(**dict(cs, wk_b=wk_t))
    assert _mismatch(o, ref)


def test_truncating_q8_0_quantiser_is_caught(monkeypatch):
    monkeypatch.setattr(O.np, "sign", np.zeros_like)   # plants rounding toward zero
    blk = np.zeros(576, np.float32)
    blk[0], blk[1] = 31.75, 0.625                     # 0.625 / 0.25 = 2.5
    codes, _ = O.quantize_q8_0(blk[None])
    assert codes[0, 1] != 3


@pytest.mark.parametrize("which", ["sign", "split_half_pairs", "exponent_i_over_d"])
def test_rope_mistakes_are_caught(monkeypatch, which):
    """A wrong rotation sign, the split-half pairing or a frequency exponent
    i/d instead of 2i/d, planted in a copy of the oracle's RoPE, fails the
    RoPE pins."""
    import tests.test_oracle_pins as P

    def bad(x, pos, b, s):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        i = np.arange(d // 2, dtype=np.float64)
        e = (i / d) if which == "exponent_i_over_d" else (2.0 * i / d)
        th = np.asarray(pos, np.float64)[..., None] * s * np.power(b, -e)
        c, sn = np.cos(th), np.sin(th)
        if which == "sign":
            sn = -sn
        if which == "split_half_pairs":
            x0, x1 = x[..., : d // 2], x[..., d // 2:]
            return np.concatenate([x0 * c - x1 * sn, x0 * sn + x1 * c], axis=-1)
        out = np.empty_like(x)
        out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * sn
        out[..., 1::2] = x[..., 0::2] * sn + x[..., 1::2] * c
        return out

    monkeypatch.setattr(O, "rope_rotate", bad)
    failed = 0
    for pin in (P.test_rope_quarter_turn_of_pair_zero_closed_form, P.test_rope_frequency_of_each_pair_closed_form):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


def test_output_projection_mistakes_are_caught(monkeypatch):
    """Summing over the wrong axis (d of W_O against the token axis) or
    dropping the head sum, planted in a copy of the oracle's projection, fails
    the projection pins."""
    import tests.test_oracle_pins as P

    for bad in (lambda o, w: np.einsum("hdD,thd->tD", np.asarray(w)[:, ::-1], np.asarray(o)),
                lambda o, w: np.einsum("hdD,thd->tD", np.asarray(w)[:1], np.asarray(o)[:, :1])):
        monkeypatch.setattr(O, "output_projection", bad)
        with pytest.raises(AssertionError):
            P.test_output_projection_matches_brute_force_loops()
