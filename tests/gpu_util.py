"""Helpers shared by the GPU parity tests: device upload of seeded inputs and
the error statistics the tolerances are written in."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from mla_latent_kv_lat_gb300 import workloads as W

# spec tolerances: max|d| / max|ref| and mean|d| / mean|ref|
TOL_BF16 = (1e-2, 2e-3)
TOL_Q8 = (3e-2, 5e-3)


def bf16_dev(vals: np.ndarray) -> torch.Tensor:
    bits = W.to_bf16(vals)[1]
    return torch.from_numpy(bits).view(torch.bfloat16).cuda()


def f16_dev(vals: np.ndarray) -> torch.Tensor:
    bits = W.to_f16(vals)[1]
    return torch.from_numpy(bits).view(torch.float16).cuda()


def dev_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def err_stats(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    return float(d.max() / np.abs(ref).max()), float(d.mean() / np.abs(ref).mean())


def assert_tol(got, ref, tol, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean = err_stats(got, ref)
    log = os.environ.get("MLA_PARITY_LOG")
    if log:                                   # optional record of every checked error, one JSON line each
        with open(log, "a") as f:
            f.write(json.dumps({"what": what, "max_rel": mx, "mean_rel": mean, "tol": list(tol)}) + "\n")
    assert mx <= tol[0] and mean <= tol[1], f"{what}: max-rel {mx:.3e} (<= {tol[0]}), mean-rel {mean:.3e} (<= {tol[1]})"
    return mx, mean


class Dev:
    """Device copies of one workload's inputs (bf16 cache packed [n, 576])."""

    def __init__(self, x: W.Inputs, q8=None):
        self.x = x
        self.q_nope = bf16_dev(x.q_nope)
        self.q_pe = bf16_dev(x.q_pe)
        self.wk_b = bf16_dev(x.wk_b)
        self.wv_b = bf16_dev(x.wv_b)
        self.kv = torch.from_numpy(x.kv_rows_bits()).view(torch.bfloat16).cuda()
        if q8 is not None:
            codes, scales = q8
            self.kv_q = torch.from_numpy(codes).cuda()
            self.kv_d = torch.from_numpy(np.ascontiguousarray(scales.T)).cuda()    # [18, n] block-major
        if x.seq_len is not None:
            self.seq_len = torch.from_numpy(x.seq_len.astype(np.int32)).cuda()
            self.seq_start = torch.from_numpy(x.seq_start.astype(np.int64)).cuda()
