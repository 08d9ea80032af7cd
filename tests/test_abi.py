"""The C-ABI library builds, loads and exports every symbol include/mla.h
declares; host-side argument checks return their status before any CUDA call
(no GPU needed)."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_lat_gb300 as mla
from mla_latent_kv_lat_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla.h")


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.load_library()


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert names == binding.declared_symbols()


def test_status_strings_and_version(lib):
    assert mla.mla_version().startswith("mla-gb300")
    for s in range(-6, 1):
        assert mla.mla_status_string(s) not in ("", "unknown status")
    assert mla.mla_status_string(42) == "unknown status"


def _dims(H=16, **kw):
    d = binding.make_dims(H)
    for k, v in kw.items():
        setattr(d, k, v)
    return ctypes.byref(d)


P = ctypes.c_void_p
GOOD = P(0x100000)          # 16-byte aligned, never dereferenced: checks fail first
ODD = P(0x100008)


def test_host_validation_rejects_bad_arguments(lib):
    assert lib.mla_absorb_q(None, GOOD, GOOD, GOOD, 4, None) == -1
    assert lib.mla_absorb_q(_dims(kv_lora_rank=256), GOOD, GOOD, GOOD, 4, None) == -2
    assert lib.mla_absorb_q(_dims(H=24), GOOD, GOOD, GOOD, 4, None) == -2
    assert lib.mla_absorb_q(_dims(H=256), GOOD, GOOD, GOOD, 4, None) == -2
    assert lib.mla_absorb_q(_dims(), None, GOOD, GOOD, 4, None) == -1
    assert lib.mla_absorb_q(_dims(), ODD, GOOD, GOOD, 4, None) == -3
    assert lib.mla_absorb_q(_dims(), GOOD, GOOD, GOOD, 0, None) == -1
    assert lib.mla_late_decompress(_dims(), GOOD, GOOD, ODD, 4, None) == -3
    # prefill: positions must stay inside the cache; the workspace holds every row as fp16
    pw = lib.mla_prefill_workspace_size(_dims(), 10)
    assert pw == (10 * 1152 + 255) // 256 * 256
    assert lib.mla_prefill_workspace_size(_dims(), 0) == 0
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 8, 3, GOOD, pw, GOOD, None, None) == -1
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 0, 0, GOOD, pw, GOOD, None, None) == -1
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 4, -1, GOOD, pw, GOOD, None, None) == -1
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 4, 0, GOOD, pw, GOOD, ODD, None) == -3
    assert lib.mla_attn_prefill(_dims(scale=0.0), GOOD, GOOD, GOOD, 10, 4, 0, GOOD, pw, GOOD, None, None) == -1
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 4, 0, GOOD, pw - 1, GOOD, None, None) == -4
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 4, 0, None, pw, GOOD, None, None) == -4
    assert lib.mla_attn_prefill(_dims(), GOOD, GOOD, GOOD, 10, 4, 0, ODD, pw, GOOD, None, None) == -3
    assert lib.mla_attn_prefill_q8_0(_dims(), GOOD, GOOD, GOOD, None, 10, 4, 0, GOOD, pw, GOOD, None, None) == -1
    # cache append: sizes, frequencies, at least one cache, the q8_0 pair together, alignment
    ra = lib.mla_rope_append
    assert ra(GOOD, GOOD, GOOD, GOOD, 0, 10000.0, 0.025, GOOD, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, GOOD, None, None, 0, 0, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 1.0, 0.025, GOOD, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.0, GOOD, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, float("nan"), GOOD, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, None, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, None, GOOD, None, 8, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, None, GOOD, GOOD, 7, 8, None) == -1
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, None, GOOD, P(0x100001), 8, 8, None) == -3
    assert ra(GOOD, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, ODD, None, None, 0, 8, None) == -3
    assert ra(None, GOOD, GOOD, GOOD, 4, 10000.0, 0.025, GOOD, None, None, 0, 8, None) == -1
    assert ra(GOOD, GOOD, ODD, GOOD, 4, 10000.0, 0.025, GOOD, None, None, 0, 8, None) == -3
    # decode: workspace size is checked on the host
    need = lib.mla_decode_workspace_size(_dims(128), 32, 32768)
    assert need > 0
    assert lib.mla_decode_workspace_size(_dims(128), 0, 32768) == 0
    assert lib.mla_attn_decode(_dims(128), GOOD, GOOD, GOOD, 100, GOOD, GOOD, 32, 32768, GOOD,
                               need - 1, GOOD, None) == -4
    assert lib.mla_attn_decode(_dims(128), GOOD, GOOD, GOOD, 100, GOOD, GOOD, 32, 32768, None,
                               need, GOOD, None) == -4
    assert lib.mla_attn_decode(_dims(128), GOOD, GOOD, GOOD, 100, GOOD, GOOD, 0, 32768, GOOD,
                               need, GOOD, None) == -1
    assert lib.mla_quantize_q8_0(GOOD, GOOD, GOOD, 10, 5, None) == -1
    assert lib.mla_quantize_q8_0(GOOD, GOOD, P(0x100001), 10, 10, None) == -3
    assert lib.mla_selftest_wait_timeout(0, None) == -1


def test_workspace_size_grows_with_batch_not_length(lib):
    # one partial per piece: at most B + G - 1 of H x 2056 bytes, G = clusters
    a = lib.mla_decode_workspace_size(_dims(128), 8, 4096)
    b = lib.mla_decode_workspace_size(_dims(128), 16, 4096)
    c = lib.mla_decode_workspace_size(_dims(128), 8, 65536)
    assert 0 < a < b and a == c
    assert b - a == 8 * 128 * 2056 and a % (128 * 2056) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()
