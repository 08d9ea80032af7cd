"""Seeded synthetic workloads for absorbed Multi-head Latent Attention.

This module only draws numbers and lays them out; it holds none of the
method's arithmetic.  Both the CPU oracle (in its tests) and the CUDA path
(tests, bench) take their inputs from here, so the two sides always see the
same values.

Shapes follow the DeepSeek MLA problem statement of the method page
("MLA matrix absorption in ik_llama.cpp", sections 1-5) and the GGUF metadata
quoted on the ik_llama.cpp PR #394 page (section 2.1: kv_lora_rank 512,
key_length 576 = 512 latent + 64 rope, value_length 512, nope 128, v 128):

* ``c_kv``  [n_rows, 512]  latent cache rows,
* ``k_pe``  [n_rows, 64]   RoPE keys, shared by every head,
* ``q_nope``[T, H, 128], ``q_pe`` [T, H, 64] queries (RoPE already applied),
* ``wk_b``  [H, 128, 512]  K up-projection (per head),
* ``wv_b``  [H, 512, 128]  V up-projection (per head),
* ``w_o``   [H, 128, D]    the output projection after the path (``make_wo``;
  D = 2048 for the Lite shape, 7168 for the V3 shape -- the two models' hidden
  sizes, which the pages do not print).

Distributions: activations N(0, 1); weights N(0, std = 1/sqrt(fan_in)) with
fan_in = 128 for wk_b and 512 for wv_b.  Every value is drawn in fp32 from one
``numpy.random.Generator(PCG64(seed))`` and rounded to bfloat16 (round to
nearest even), so each tensor is exactly representable in bf16.  Draw order:
(decode only: the cache lengths), c_kv, k_pe, q_nope, q_pe, wk_b, wv_b.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

KV_LORA_RANK = 512
QK_ROPE = 64
QK_NOPE = 128
V_HEAD = 128
ROW = KV_LORA_RANK + QK_ROPE          # 576 values per latent-cache row
DEFAULT_SCALE = 1.0 / math.sqrt(QK_NOPE + QK_ROPE)


def to_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round fp32 ``x`` to bfloat16 (nearest, ties to even).

    Returns ``(values, bits)``: the rounded values as float32 and their raw
    16-bit patterns as uint16 (what a device bf16 buffer holds).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    bits = u.astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return vals, bits


def to_f16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round fp32 ``x`` to IEEE half (nearest, ties to even): ``(values, bits)``."""
    h = np.ascontiguousarray(x, dtype=np.float32).astype(np.float16)
    return h.astype(np.float32), h.view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named workload: a prefill chunk or a batch of decode queries."""
    name: str
    kind: str                 # "prefill" | "decode" | "append" (new tokens into the cache)
    n_head: int
    cache: str                # "bf16" | "q8_0"
    T: int = 0                # prefill: query tokens
    q_pos0: int = 0           # prefill: position of query 0
    n_kv: int = 0             # prefill: cache rows (positions 0..n_kv-1)
    B: int = 0                # decode: sequences
    len_lo: int = 0           # decode: cache length range, inclusive
    len_hi: int = 0
    hidden: int = 0           # model width D of the output projection wo [H*128, D]
    describe: str = ""

    @property
    def scale(self) -> float:
        return DEFAULT_SCALE


WORKLOADS = {
    "lite_t256": Workload(
        "lite_t256", "prefill", 16, "bf16", T=256, q_pos0=0, n_kv=256, hidden=2048,
        describe="DeepSeek-Lite shape, 16 heads, 256-token causal prefill over its own 256-row cache"),
    "lite_t4096": Workload(
        "lite_t4096", "prefill", 16, "bf16", T=4096, q_pos0=0, n_kv=4096, hidden=2048,
        describe="DeepSeek-Lite shape, 16 heads, 4096-token causal prefill"),
    "v3_chunk8192_at32768": Workload(
        "v3_chunk8192_at32768", "prefill", 128, "bf16", T=8192, q_pos0=32768, n_kv=40960, hidden=7168,
        describe="DeepSeek-V3 shape, 128 heads, 8192-query chunked prefill at positions "
                 "32768..40959 over a 40960-row latent cache"),
    "v3_decode_b32": Workload(
        "v3_decode_b32", "decode", 128, "bf16", B=32, len_lo=4096, len_hi=32768, hidden=7168,
        describe="DeepSeek-V3 shape decode, 32 sequences, one query each, "
                 "cache lengths uniform in [4096, 32768]"),
    "v3_q8_chunk8192_at90112": Workload(
        "v3_q8_chunk8192_at90112", "prefill", 128, "q8_0", T=8192, q_pos0=90112, n_kv=98304, hidden=7168,
        describe="DeepSeek-V3 shape, q8_0 latent cache, 8192-query causal prefill at "
                 "positions 90112..98303 over 98304 rows"),
    "v3_q8_decode_b8": Workload(
        "v3_q8_decode_b8", "decode", 128, "q8_0", B=8, len_lo=98304, len_hi=98304, hidden=7168,
        describe="DeepSeek-V3 shape, q8_0 latent cache, 8 sequences decoding at length 98304"),
    # The step before the path: T new tokens' rows (RoPE applied) into a bf16
    # and a q8_0 cache of n_kv rows, at distinct random slots -- the fill of
    # the 98304-row q8_0 cache of the V3 q8_0 workloads.
    "v3_cache_append_98304": Workload(
        "v3_cache_append_98304", "append", 128, "bf16+q8_0", T=98304, n_kv=98304,
        describe="cache append: 98304 new tokens' rows (RoPE on the 64-d part) into a bf16 and a "
                 "q8_0 latent cache of 98304 rows at random slots"),
}


@dataclasses.dataclass
class Inputs:
    """Host-side tensors of one workload; every float array holds bf16 values."""
    wl: Workload
    c_kv: np.ndarray          # [n_rows, 512] float32 (bf16 values)
    k_pe: np.ndarray          # [n_rows, 64]
    q_nope: np.ndarray        # [T or B, H, 128]
    q_pe: np.ndarray          # [T or B, H, 64]
    wk_b: np.ndarray          # [H, 128, 512]
    wv_b: np.ndarray          # [H, 512, 128]
    seq_len: Optional[np.ndarray] = None    # decode: [B] int32
    seq_start: Optional[np.ndarray] = None  # decode: [B] int64 row offsets

    @property
    def n_rows(self) -> int:
        return self.c_kv.shape[0]

    def q_pos(self) -> np.ndarray:
        """Position of every query row (prefill: q_pos0 + t; decode: len - 1)."""
        if self.wl.kind == "prefill":
            return self.wl.q_pos0 + np.arange(self.wl.T, dtype=np.int64)
        return self.seq_len.astype(np.int64) - 1

    def kv_rows_bits(self) -> np.ndarray:
        """The packed bf16 cache [n_rows, 576]: latent 0..511, rope 512..575."""
        return to_bf16(np.concatenate([self.c_kv, self.k_pe], axis=1))[1]


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std) fp32 draws rounded to bf16 (values as float32)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16(x)[0]


def normal_f16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std) fp32 draws rounded to fp16 (values as float32)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_f16(x)[0]


def decode_lengths(wl: Workload, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(wl.len_lo, wl.len_hi + 1, size=wl.B, dtype=np.int64).astype(np.int32)


def make_inputs(wl: Workload | str, seed: int = 0, *, n_head: Optional[int] = None,
                T: Optional[int] = None, q_pos0: Optional[int] = None,
                n_kv: Optional[int] = None, lengths: Optional[np.ndarray] = None) -> Inputs:
    """Draw one workload's inputs.  Keyword overrides build smaller variants
    with the same distributions (parity tests at sizes the oracle finishes)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    over = {}
    if n_head is not None:
        over["n_head"] = n_head
    if T is not None:
        over["T"] = T
    if q_pos0 is not None:
        over["q_pos0"] = q_pos0
    if n_kv is not None:
        over["n_kv"] = n_kv
    if lengths is not None:
        lengths = np.asarray(lengths, dtype=np.int32)
        over.update(B=int(lengths.size), len_lo=int(lengths.min()), len_hi=int(lengths.max()))
    if over:
        wl = dataclasses.replace(wl, name=wl.name + "_var", **over)
    rng = np.random.default_rng(seed)
    H = wl.n_head
    seq_len = seq_start = None
    if wl.kind == "decode":
        if lengths is None:
            lengths = rng.integers(wl.len_lo, wl.len_hi + 1, size=wl.B, dtype=np.int64).astype(np.int32)
        seq_len = lengths
        seq_start = np.zeros(wl.B, dtype=np.int64)
        seq_start[1:] = np.cumsum(seq_len.astype(np.int64))[:-1]
        n_rows = int(seq_len.astype(np.int64).sum())
        nq = wl.B
    else:
        if wl.q_pos0 + wl.T > wl.n_kv:
            raise ValueError("prefill queries must lie inside the cache")
        n_rows = wl.n_kv
        nq = wl.T
    c_kv = normal_bf16(rng, (n_rows, KV_LORA_RANK))
    k_pe = normal_bf16(rng, (n_rows, QK_ROPE))
    q_nope = normal_bf16(rng, (nq, H, QK_NOPE))
    q_pe = normal_bf16(rng, (nq, H, QK_ROPE))
    wk_b = normal_bf16(rng, (H, QK_NOPE, KV_LORA_RANK), 1.0 / math.sqrt(QK_NOPE))
    wv_b = normal_bf16(rng, (H, KV_LORA_RANK, V_HEAD), 1.0 / math.sqrt(KV_LORA_RANK))
    return Inputs(wl, c_kv, k_pe, q_nope, q_pe, wk_b, wv_b, seq_len, seq_start)


def make_wo(n_head: int, hidden: int, seed: int = 0) -> np.ndarray:
    """The output projection wo as [H, 128, hidden] (row-major [H*128, hidden]):
    N(0, std = 1/sqrt(H*128)) rounded to bf16, from its own generator (seeded
    with (seed, 1)), so that drawing it changes none of the other inputs."""
    rng = np.random.default_rng([seed, 1])
    return normal_bf16(rng, (n_head, V_HEAD, hidden), 1.0 / math.sqrt(n_head * V_HEAD))


def sample_rows(n: int, k: int, seed: int = 0, must: tuple = ()) -> np.ndarray:
    """``k`` distinct row indices in [0, n), always holding ``must`` (clipped)."""
    rng = np.random.default_rng(seed + 7919)
    base = set(int(m) for m in must if 0 <= m < n)
    pool = rng.permutation(n)
    out = list(base)
    for r in pool:
        if len(out) >= min(k, n):
            break
        if int(r) not in base:
            out.append(int(r))
    return np.array(sorted(out), dtype=np.int64)


# ---------------------------------------------------------------------------
# New tokens for the cache-append step (mla_rope_append)
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class AppendInputs:
    c_kv: np.ndarray      # [n, 512] bf16 values as float32
    k_pe: np.ndarray      # [n, 64]  bf16 values as float32 (not yet rotated)
    pos: np.ndarray       # [n] int32 positions
    slot: np.ndarray      # [n] int64 distinct cache rows in [0, n_rows)
    n_rows: int


def make_append_inputs(n: int, n_rows: int, seed: int = 0, max_pos: int = 98304) -> AppendInputs:
    """n new tokens with N(0,1) bf16 latent and RoPE parts (the distributions
    of the cache rows in every workload), positions uniform in [0, max_pos)
    plus the two ends, and distinct slots drawn from the cache's n_rows rows."""
    assert 1 <= n <= n_rows
    rng = np.random.default_rng(seed)
    c_kv = to_bf16(rng.standard_normal((n, KV_LORA_RANK), dtype=np.float32))[0]
    k_pe = to_bf16(rng.standard_normal((n, QK_ROPE), dtype=np.float32))[0]
    pos = rng.integers(0, max_pos, n).astype(np.int32)
    pos[0] = 0
    if n > 1:
        pos[-1] = max_pos - 1
    slot = rng.permutation(n_rows)[:n].astype(np.int64)
    return AppendInputs(c_kv, k_pe, pos, slot, n_rows)
