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
