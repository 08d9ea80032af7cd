"""CPU oracle for Multi-head Latent Attention on a compressed latent KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or
run anything here.  The CUDA library never calls it and shares no code with
it; the two meet only in the seeded inputs of ``workloads.py``.

Everything is plain numpy in float64 (inputs are bf16 values held in float32
and widened on entry).  Library matmuls serve as steps; there is no blocking,
fusion or reordering beyond what each definition states.

Sources (web pages, cited by title and section):

* [MLA] "MLA matrix absorption in ik_llama.cpp" (czykbl.com/news/93068):
  sec. 1 (decompression k = W^UK c, v = W^UV c), sec. 2 (associativity),
  sec. 3 (K absorption), sec. 4 (V absorption / late decompression, einsums
  ``bhql,blc->bhqc`` and ``bhqc,hdc->bhqd``), sec. 5 (split scores: RoPE part
  plus latent part), sec. 7 (cache size and FLOP table), sec. 8.1 (q8_0 cache).
* [PR394] "ik_llama.cpp PR #394 mainline DeepSeek GGUF support"
  (czykbl.com/news/94940): sec. 2.1 (kv_lora_rank 512, key_length 576,
  value_length 512, nope 128, v 128, rope 64), sec. 3.2 (wk_b / wv_b layouts).
* [KVRM] "ik_llama.cpp discussion #586 slow KV cache rm" (trdm.cn/news/546512):
  the log line giving the q8_0 latent cache size at n_ctx 98304, and the
  context log of the same run (sec. "混合卸载配置解读": freq_base 10000.0,
  freq_scale 0.025).
* [KVC] "llama.cpp KV Cache 与注意力机制：环形缓冲到 Flash Attention"
  (borninfreedom.github.io/posts/2026/07/blog-post-4): sec. 2.2 (new tokens
  are written into cache slots found for them), sec. 2.3 (keys are rotated
  by ``ggml_rope_ext`` with n_rot dimensions).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force on tiny inputs, invariants, the pages' printed
numbers).  No function is "parity unpinned".
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# Dimensions of the DeepSeek MLA layer ([PR394] sec. 2.1)
# ---------------------------------------------------------------------------
KV_LORA_RANK = 512       # latent width of c_kv
QK_ROPE = 64             # RoPE part of every key / query
QK_NOPE = 128            # non-RoPE part of every query / decompressed key, per head
V_HEAD = 128             # value width per head
Q8_BLOCK = 32            # q8_0 block: 32 int8 codes + one fp16 scale ([MLA] sec. 8.1)


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The un-absorbed definition ([MLA] sec. 1, with the score split of sec. 3/5)
# ---------------------------------------------------------------------------
def decompress_head(c_kv: np.ndarray, wk_b_h: np.ndarray, wv_b_h: np.ndarray):
    """Explicit decompression of every cache row for one head ([MLA] sec. 1).

    k_nope[j, d] = sum_c wk_b_h[d, c] * c_kv[j, c]     (W^UK c,  128-d)
    v[j, e]      = sum_c wv_b_h[c, e] * c_kv[j, c]     (W^UV c,  128-d)

    ``wk_b_h`` is [128, 512] (row d, column c); ``wv_b_h`` is [512, 128].
    """
    c = _f64(c_kv)
    k_nope = c @ _f64(wk_b_h).T
    v = c @ _f64(wv_b_h)
    return k_nope, v


def attention_unabsorbed(q_nope, q_pe, c_kv, k_pe, wk_b, wv_b, q_pos, scale: float,
                         heads: Optional[Sequence[int]] = None):
    """Standard causal attention on explicitly decompressed keys and values.

    For query row t (position ``q_pos[t]``) and head h:
      Q = [q_nope[t,h], q_pe[t,h]]            (192-d)
      K_j = [k_nope[j,h], k_pe[j]]            (192-d, k_pe shared by all heads)
      s_j = scale * Q.K_j  for j <= q_pos[t], excluded otherwise
      p = softmax(s);  o[t,h] = sum_j p_j v[j,h]

    Cache row j holds position j.  Returns ``(o [T, nh, 128], lse [T, nh])``
    with lse = log sum_j exp(s_j) (natural log), over the selected heads.
    """
    q_nope = _f64(q_nope)
    q_pe = _f64(q_pe)
    k_pe = _f64(k_pe)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    T, H, _ = q_nope.shape
    heads = list(range(H)) if heads is None else list(heads)
    n_vis = int(q_pos.max()) + 1
    c = _f64(c_kv)[:n_vis]
    kp = k_pe[:n_vis]
    j = np.arange(n_vis)
    visible = j[None, :] <= q_pos[:, None]                 # [T, n_vis]
    o = np.empty((T, len(heads), np.shape(wv_b)[2]))
    lse = np.empty((T, len(heads)))
    for hi, h in enumerate(heads):
        k_nope, v = decompress_head(c, wk_b[h], wv_b[h])
        Q = np.concatenate([q_nope[:, h, :], q_pe[:, h, :]], axis=1)      # [T, 192]
        K = np.concatenate([k_nope, kp], axis=1)                          # [n_vis, 192]
        s = scale * (Q @ K.T)
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        o[:, hi, :] = (e / den) @ v
        lse[:, hi] = (m + np.log(den))[:, 0]
    return o, lse


# ---------------------------------------------------------------------------
# The absorbed rearrangement ([MLA] sec. 3-5): exact up to rounding order
# ---------------------------------------------------------------------------
def absorb_q(q_nope, wk_b):
    """K absorption ([MLA] sec. 3): q_lat[t,h,c] = sum_d q_nope[t,h,d] * wk_b[h,d,c]."""
    return np.einsum("thd,hdc->thc", _f64(q_nope), _f64(wk_b), optimize=True)


def attention_latent(q_lat, q_pe, c_kv, k_pe, q_pos, scale: float):
    """Split-score causal attention in latent space ([MLA] sec. 4-5).

    s[t,h,j] = scale * (q_pe[t,h].k_pe[j] + q_lat[t,h].c_kv[j]),  j <= q_pos[t]
    o_lat[t,h] = sum_j softmax(s)[j] * c_kv[j]        (512-d, before W^UV)
    Returns ``(o_lat [T, H, 512], lse [T, H])``.
    """
    q_lat = _f64(q_lat)
    q_pe = _f64(q_pe)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    n_vis = int(q_pos.max()) + 1
    c = _f64(c_kv)[:n_vis]
    kp = _f64(k_pe)[:n_vis]
    T, H, _ = q_lat.shape
    visible = np.arange(n_vis)[None, :] <= q_pos[:, None]
    o_lat = np.empty((T, H, c.shape[1]))
    lse = np.empty((T, H))
    for h in range(H):
        s = scale * (q_pe[:, h, :] @ kp.T + q_lat[:, h, :] @ c.T)
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        o_lat[:, h, :] = (e / den) @ c
        lse[:, h] = (m + np.log(den))[:, 0]
    return o_lat, lse


def late_decompress(o_lat, wv_b):
    """Late V decompression ([MLA] sec. 4): o[t,h,e] = sum_c o_lat[t,h,c] * wv_b[h,c,e]."""
    return np.einsum("thc,hce->the", _f64(o_lat), _f64(wv_b), optimize=True)


def output_projection(o, w_o):
    """The step after the path ([MLA] sec. 4, the einsum ``hdD,bhqd->bqD``):
    u[t, D] = sum_h sum_d w_o[h, d, D] * o[t, h, d], with o the per-head output
    [T, H, 128] of late decompression and w_o [H, 128, hidden] (the pages' own
    layout of W_O).  float64."""
    return np.einsum("hdD,thd->tD", _f64(w_o), _f64(o), optimize=True)


def projected_weights(wv_b, w_o):
    """W_O folded into W_UV per head ([MLA] sec. 6, the offline pre-absorption
    the page weighs and rejects as slower): m[h, c, D] = sum_d wv_b[h, c, d] *
    w_o[h, d, D], so that u = sum_h o_lat[:, h, :] . m[h]."""
    return np.einsum("hcd,hdD->hcD", _f64(wv_b), _f64(w_o), optimize=True)


def attention_absorbed(q_nope, q_pe, c_kv, k_pe, wk_b, wv_b, q_pos, scale: float):
    """The whole absorbed chain: absorb -> latent attention -> late decompression."""
    q_lat = absorb_q(q_nope, wk_b)
    o_lat, lse = attention_latent(q_lat, q_pe, c_kv, k_pe, q_pos, scale)
    return late_decompress(o_lat, wv_b), o_lat, lse


# ---------------------------------------------------------------------------
# Decode: one query per sequence at position len-1, over that sequence's rows
# ---------------------------------------------------------------------------
def decode_unabsorbed(q_nope, q_pe, c_kv, k_pe, wk_b, wv_b, seq_start, seq_len, scale: float,
                      heads: Optional[Sequence[int]] = None, seqs: Optional[Sequence[int]] = None):
    """Per sequence b: the query q[b] sits at position len_b - 1 and attends the
    len_b rows starting at row ``seq_start[b]``.  Returns o [nb, nh, 128]."""
    seqs = list(range(len(seq_len))) if seqs is None else list(seqs)
    outs = []
    for b in seqs:
        s0, n = int(seq_start[b]), int(seq_len[b])
        o, _ = attention_unabsorbed(q_nope[b:b + 1], q_pe[b:b + 1], c_kv[s0:s0 + n], k_pe[s0:s0 + n],
                                    wk_b, wv_b, [n - 1], scale, heads=heads)
        outs.append(o[0])
    return np.stack(outs)


def decode_latent(q_lat, q_pe, c_kv, k_pe, seq_start, seq_len, scale: float,
                  seqs: Optional[Sequence[int]] = None):
    """Latent-space decode (absorbed form); returns o_lat [nb, H, 512], lse [nb, H]."""
    seqs = list(range(len(seq_len))) if seqs is None else list(seqs)
    ol, ls = [], []
    for b in seqs:
        s0, n = int(seq_start[b]), int(seq_len[b])
        o_lat, lse = attention_latent(q_lat[b:b + 1], q_pe[b:b + 1], c_kv[s0:s0 + n], k_pe[s0:s0 + n],
                                      [n - 1], scale)
        ol.append(o_lat[0])
        ls.append(lse[0])
    return np.stack(ol), np.stack(ls)


# ---------------------------------------------------------------------------
# q8_0 latent cache ([MLA] sec. 8.1 "MLA with Q8_0 KV cache"; [KVRM] cache size)
# ---------------------------------------------------------------------------
def quantize_q8_0(x: np.ndarray):
    """Quantise rows of 576 values into 18 blocks of 32 int8 codes + one fp16 scale.

    The pages fix the block format (32 codes + fp16 scale = 34 bytes, which is
    what reproduces the 3499.88 MiB cache of [KVRM]) but not the rounding.
    Reading adopted: per block, amax = max|x|; d = amax / 127 in fp32;
    q = round-half-away-from-zero(x / d) in fp32, clamped to [-127, 127]
    (q = 0 when amax = 0); the stored scale is fp16(d).  All decisions are
    taken in fp32, the precision of the device quantiser.

    Returns ``(codes int8 [n, 576], scales float16 [n, 18])``.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, width = x.shape
    assert width % Q8_BLOCK == 0
    xb = x.reshape(n, width // Q8_BLOCK, Q8_BLOCK)
    amax = np.abs(xb).max(axis=2)                                   # fp32
    d = (amax / np.float32(127.0)).astype(np.float32)               # fp32 division, RN
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    y = (xb / safe[:, :, None]).astype(np.float32)                  # fp32 division, RN
    t = np.trunc(y)
    frac = np.abs(y - t)                                            # exact for |y| < 2^23
    r = t + np.sign(y) * (frac >= np.float32(0.5))
    r = np.clip(r, -127, 127)
    r = np.where(d[:, :, None] > 0, r, 0)
    codes = r.astype(np.int8).reshape(n, width)
    return codes, d.astype(np.float16)


# ---------------------------------------------------------------------------
# The step before the path: new tokens' rows into the latent cache
# ([MLA] sec. 3: the RoPE part is rotated by position and kept apart from the
# latent part; [KVC] sec. 2.2-2.3; [KVRM] freq_base / freq_scale)
# ---------------------------------------------------------------------------
def rope_rotate(x: np.ndarray, pos, freq_base: float, freq_scale: float) -> np.ndarray:
    """Rotary position encoding of the last dimension (d = 64 for k_pe).

    Readings (the pages name ``ggml_rope_ext`` with n_rot = 64, freq_base and
    freq_scale, but not the pairing or any extension of the frequencies):
    dimensions (2i, 2i+1) form pair i (ggml's default, "normal" mode) and are
    rotated by the angle theta_i = pos * freq_scale * freq_base^(-2i/d):
    (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).  No other scaling.
    ``pos`` broadcasts against x's leading dimensions.  float64.
    """
    x = _f64(x)
    d = x.shape[-1]
    assert d % 2 == 0
    i = np.arange(d // 2, dtype=np.float64)
    theta = _f64(pos)[..., None] * float(freq_scale) * np.power(float(freq_base), -2.0 * i / d)
    c, s = np.cos(theta), np.sin(theta)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def cache_rows(c_kv_new: np.ndarray, k_pe_new: np.ndarray, pos, freq_base: float, freq_scale: float) -> np.ndarray:
    """The cache rows of new tokens: [c_kv (512, as given) | RoPE(k_pe, pos) (64)],
    float64 (the cache stores them in its element type: bf16, or q8_0 via
    ``quantize_q8_0``)."""
    return np.concatenate([_f64(c_kv_new), rope_rotate(k_pe_new, pos, freq_base, freq_scale)], axis=-1)


def dequantize_q8_0(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """x = fp16(d_b) * q_i for element i of block b (float64, exact)."""
    n, width = codes.shape
    q = codes.astype(np.float64).reshape(n, width // Q8_BLOCK, Q8_BLOCK)
    return (q * scales.astype(np.float64)[:, :, None]).reshape(n, width)


# ---------------------------------------------------------------------------
# Accounting ([MLA] sec. 7 table; [KVRM] cache size)
# ---------------------------------------------------------------------------
def latent_row_bytes(elem_bytes: int = 2) -> int:
    """Bytes of one cached token in the latent cache: c_kv (512) + k_pe (64)."""
    return (KV_LORA_RANK + QK_ROPE) * elem_bytes


def q8_0_row_bytes() -> int:
    """One 576-value row in q8_0: 18 blocks of (32 int8 + 2-byte fp16 scale)."""
    nb = (KV_LORA_RANK + QK_ROPE) // Q8_BLOCK
    return nb * (Q8_BLOCK + 2)


def decompressed_token_bytes(n_head: int, elem_bytes: int = 2) -> int:
    """Bytes of one token's decompressed K (nope 128 + rope 64) and V (128), all heads."""
    return n_head * (QK_NOPE + QK_ROPE + V_HEAD) * elem_bytes


def flops_per_pair_decompressed(n_head: int) -> int:
    """Attention FLOPs per (query, key) pair on a decompressed cache: 2*192 + 2*128 per head."""
    return n_head * (2 * (QK_NOPE + QK_ROPE) + 2 * V_HEAD)


def flops_per_token_decompress(n_head: int) -> int:
    """Decompressing one cached token for all heads: 2 * 512 * (128 + 128) * n_head."""
    return 2 * KV_LORA_RANK * (QK_NOPE + V_HEAD) * n_head


def flops_per_pair_absorbed(n_head: int) -> int:
    """Absorbed attention FLOPs per (query, key) pair: 2*576 (scores) + 2*512 (latent sum) per head."""
    return n_head * (2 * (KV_LORA_RANK + QK_ROPE) + 2 * KV_LORA_RANK)


def causal_pairs(T: int, q_pos0: int) -> int:
    """Visible (query, key) pairs of a causal chunk: query t sees q_pos0 + t + 1 keys."""
    return T * q_pos0 + T * (T + 1) // 2
