"""Benchmark of the absorbed-MLA hot path on one GB300 (or N replicas).

A step is one pass of the whole path over one batch of the workload:
absorb (wk_b into the query) -> causal latent attention -> late
decompression (wv_b); decode workloads add the split-KV combine and q8_0
workloads dequantise the cache inside the attention kernel.  Inputs are the
seeded synthetic tensors of ``workloads.py`` (no dataset), resident in HBM
when the timed region starts.  L2 (129 MB) is flushed by writing a 512 MB
buffer before every timed step; only the step itself is inside the CUDA events.

The JSON line's headline is the DeepSeek-V3-shape 8192-query chunk at
position 32768 (the largest prefill that fits the bf16 cache workloads); every
other workload follows under "secondary", each with its own roofline of the
dominant kernel and its end-to-end number (host buffers, copies inside the
timed region).

``--impl reference`` times the CPU oracle (the un-absorbed definition in
numpy fp64) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_latent_kv_lat_gb300 import workloads as W  # noqa: E402

METRIC = "MLA attn TFLOP/s (prefill) & HBM GB/s (decode) on 1 GB300, % of roofline"
# The headline line: the largest single-GPU prefill (DeepSeek-V3 shape, an
# 8192-query chunk at position 32768).  Every other workload is measured too,
# each as a secondary entry with its own roofline and end-to-end number.
DEFAULT_WORKLOAD = "v3_chunk8192_at32768"
# "<workload>:materialized" is the same chunk through the materialised
# prefill (per-head K/V decompressed, then standard attention: the pp_opt
# path); "<workload>:projected" appends the output projection wo to the
# absorbed path (late decompression to fp16, then u = o . w_o with w_o
# converted once from the model's bf16 to fp16 before any step).
SECONDARY_WORKLOADS = ["lite_t4096", "lite_t256", "v3_decode_b32", "v3_q8_chunk8192_at90112", "v3_q8_decode_b8",
                       "v3_cache_append_98304", "v3_chunk8192_at32768:materialized", "lite_t4096:materialized",
                       "v3_q8_chunk8192_at90112:materialized", "v3_chunk8192_at32768:projected",
                       "lite_t4096:projected"]
FLOP_PER_PAIR_HEAD = 2 * 576 + 2 * 512          # scores (576-d) + latent weighted sum (512-d)
# sources whose hash dates the ncu traffic recorded for each kernel
KERNEL_SOURCES = {"attn_tc_kernel": ["attn_tc.cu", "tc.cuh", "common.cuh", "kernels.cuh"],
                  "rope_append_kernel": ["append.cu", "append.cuh", "common.cuh"],
                  "pp_attn_tc_kernel": ["materialize.cu", "tc.cuh", "common.cuh", "kernels.cuh"],
                  "wo_gemm_tc_kernel": ["wo_tc.cu", "tc.cuh", "common.cuh", "kernels.cuh"]}


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------
def attn_flops(wl: W.Workload, x: W.Inputs) -> float:
    if wl.kind == "prefill":
        pairs = wl.T * wl.q_pos0 + wl.T * (wl.T + 1) // 2
    else:
        pairs = int(x.seq_len.astype(np.int64).sum())
    return float(pairs) * wl.n_head * FLOP_PER_PAIR_HEAD


def decode_bytes(wl: W.Workload, x: W.Inputs) -> float:
    row = 576 * 2 if wl.cache == "bf16" else 576 + 18 * 2
    q = wl.B * wl.n_head * (512 + 64) * 2
    o = wl.B * wl.n_head * 512 * 2
    return float(x.seq_len.astype(np.int64).sum()) * row + q + o


# bytes per appended token: c_kv + k_pe in (bf16), position and slot, the bf16
# row and the q8_0 row (codes + 18 fp16 scales) out
APPEND_TOKEN_BYTES = (512 + 64) * 2 + 4 + 8 + 576 * 2 + 576 + 18 * 2


def append_bytes(wl: W.Workload) -> float:
    return float(wl.T) * APPEND_TOKEN_BYTES


# the materialised prefill's own work: 2*192 + 2*128 FLOPs per visible pair and
# head, plus decompressing every row it reads (512 -> 128 + 128 per head)
FLOP_PER_PAIR_HEAD_MATERIALIZED = 2 * 192 + 2 * 128


def materialized_flops(wl: W.Workload) -> float:
    pairs = wl.T * wl.q_pos0 + wl.T * (wl.T + 1) // 2
    rows = wl.q_pos0 + wl.T
    return float(pairs) * wl.n_head * FLOP_PER_PAIR_HEAD_MATERIALIZED + float(rows) * wl.n_head * 2 * 512 * 256


def wo_flops(wl: W.Workload) -> float:
    return 2.0 * wl.T * wl.n_head * 128 * wl.hidden


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_hash(kernel: str = "attn_tc_kernel") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, "mla_latent_kv_lat_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p)).get(f"{kernel}:{workload}")
    except Exception:
        return None
    if not rec or rec.get("kernel_hash") != kernel_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def _samples(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def _wait_for(self, n: int, limit_s: float):
        t0 = time.perf_counter()
        while self._samples() < n and time.perf_counter() - t0 < limit_s:
            time.sleep(0.02)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        if self.proc is not None:
            # a timed region shorter than the 200 ms period is still bracketed
            # by a sample before it and one after it
            self._wait_for(1, 3.0)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self._wait_for(self._samples() + 1, 1.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def setup_append(wl, torch):
    import mla_latent_kv_lat_gb300 as mla
    a = W.make_append_inputs(wl.T, wl.n_kv)
    d = {"c_kv": torch.from_numpy(W.to_bf16(a.c_kv)[1]).view(torch.bfloat16).cuda(),
         "k_pe": torch.from_numpy(W.to_bf16(a.k_pe)[1]).view(torch.bfloat16).cuda(),
         "pos": torch.from_numpy(a.pos).cuda(), "slot": torch.from_numpy(a.slot).cuda()}
    caches = {"kv": torch.zeros(wl.n_kv, 576, dtype=torch.bfloat16, device="cuda"),
              "kv_q": torch.zeros(wl.n_kv, 576, dtype=torch.int8, device="cuda"),
              "kv_d": torch.zeros(18, wl.n_kv, dtype=torch.float16, device="cuda")}

    def step(stream=None, ev=None):
        if ev:
            ev[0].record()
        mla.mla_rope_append(d["c_kv"], d["k_pe"], d["pos"], d["slot"], stream=stream, **caches)
        if ev:
            ev[1].record()
    return wl, a, d, caches, step, 1


def setup_variant(name, variant, torch):
    """The materialised prefill (one call: prep, decompression, attention) or
    the absorbed path with the output projection; the events `ev` bracket the
    materialised call, or the projection alone."""
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import pipeline as P
    wl = W.WORKLOADS[name]
    x = W.make_inputs(wl)

    def dev(a):
        return torch.from_numpy(W.to_bf16(a)[1]).view(torch.bfloat16).cuda()

    d = {"q_nope": dev(x.q_nope), "q_pe": dev(x.q_pe), "wk_b": dev(x.wk_b), "wv_b": dev(x.wv_b)}
    kv = torch.from_numpy(x.kv_rows_bits()).view(torch.bfloat16).cuda()
    T, H = wl.T, wl.n_head
    if variant == "materialized":
        if wl.cache == "q8_0":
            n = kv.shape[0]
            d["kv_q"] = torch.empty(n, 576, dtype=torch.int8, device="cuda")
            d["kv_d"] = torch.empty(18, n, dtype=torch.float16, device="cuda")
            mla.mla_quantize_q8_0(kv, d["kv_q"], d["kv_d"])     # the cache producer, outside the timing
            del kv
        else:
            d["kv"] = kv
        out = torch.empty(T, H, 128, dtype=torch.float32, device="cuda")
        ws = torch.empty(mla.mla_prefill_materialized_workspace_size(H, T, wl.q_pos0), dtype=torch.uint8,
                         device="cuda")

        def step_io(dv, o, stream=None):
            if wl.cache == "q8_0":
                mla.mla_attn_prefill_materialized_q8_0(dv["q_nope"], dv["q_pe"], dv["kv_q"], dv["kv_d"], dv["wk_b"],
                                                       dv["wv_b"], wl.q_pos0, o, workspace=ws, stream=stream)
            else:
                mla.mla_attn_prefill_materialized(dv["q_nope"], dv["q_pe"], dv["kv"], dv["wk_b"], dv["wv_b"],
                                                  wl.q_pos0, o, workspace=ws, stream=stream)

        def step(stream=None, ev=None):
            if ev:
                ev[0].record()
            step_io(d, out, stream)
            if ev:
                ev[1].record()
        return wl, x, d, (out, ws, step_io), step, 3 if wl.cache == "q8_0" else 2   # (staging,) decompression, attention
    d["kv"] = kv
    w_o = dev(W.make_wo(H, wl.hidden))
    d["w_o"] = torch.empty(w_o.shape, dtype=torch.float16, device="cuda")
    mla.mla_convert_bf16_to_f16(w_o, d["w_o"])        # weight preparation, once, outside every step
    del w_o
    bufs = P.prefill_buffers(T, H, n_kv=x.n_rows)
    pb = P.project_buffers(T, H, wl.hidden)

    def step(stream=None, ev=None):
        mla.mla_absorb_q(d["q_nope"], d["wk_b"], bufs.q_lat, stream=stream)
        mla.mla_attn_prefill(bufs.q_lat, d["q_pe"], d["kv"], wl.q_pos0, bufs.o_lat, stream=stream,
                             workspace=bufs.workspace)
        mla.mla_late_decompress_f16(bufs.o_lat, d["wv_b"], pb.o16, stream=stream)
        if ev:
            ev[0].record()
        mla.mla_output_project(pb.o16, d["w_o"], pb.u, stream=stream)
        if ev:
            ev[1].record()
    return wl, x, d, (bufs, pb), step, 5


def measure_variant(args, torch, full, flush, pk, pk_kind, world=1):
    name, variant = full.split(":")
    wl, x, d, bufs, step, launches = setup_variant(name, variant, torch)
    torch.cuda.synchronize()
    step_ms, ev_ms = time_steps(torch, step, args.steps, args.warmup, flush)
    ms = sum(step_ms) / len(step_ms)
    kms = sum(ev_ms) / len(ev_ms)
    peak = pk["bf16_tflops"]
    out = {"workload": full, "ms_per_step": round(ms, 4), "tokens_per_s": round(wl.T * world / (ms * 1e-3), 1),
           "gpu_launches": launches * args.steps}
    if variant == "materialized":
        own = materialized_flops(wl) / (kms * 1e-3) / 1e12
        out.update({"value": round(materialized_flops(wl) * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "value_of": "own work: pairs x H x 640 + rows x H x 262144 (decompression)",
                    "absorbed_equiv_tflops": round(attn_flops(wl, x) * world / (ms * 1e-3) / 1e12, 3),
                    "roofline": {"bound": "tensor", "achieved": round(own, 3), "peak": peak, "unit": "TFLOP/s",
                                 "frac": round(own / peak, 4), "peak_kind": f"{pk_kind} bf16 dense, burst",
                                 "kernel": "pp_decompress_tc_kernel+pp_attn_tc_kernel",
                                 "attn_ms": round(kms, 4),
                                 "traffic": recorded_traffic("pp_attn_tc_kernel", full),
                                 "traffic_kernel": "pp_attn_tc_kernel (the call's dominant kernel)"}})
        ms_e, h2d, d2h = e2e_overlapped(args, torch, d, bufs[0], bufs[2])
        out["e2e"] = {"value": round(materialized_flops(wl) / (ms_e * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                      "ms_per_step": round(ms_e, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "copies": "overlapped with the neighbouring steps (copy stream, two buffer sets)"}
    else:
        tf = wo_flops(wl) / (kms * 1e-3) / 1e12
        out.update({"value": round(attn_flops(wl, x) * world / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "value_of": "absorbed attention FLOPs per step, the step now ending with u = o . w_o",
                    "hidden": wl.hidden,
                    "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": peak, "unit": "TFLOP/s",
                                 "frac": round(tf / peak, 4),
                                 "peak_kind": f"{pk_kind} bf16 dense, burst (fp16 MMA: the same nominal rate)",
                                 "kernel": "wo_gemm_tc_kernel", "attn_ms": round(kms, 4),
                                 "traffic": recorded_traffic("wo_gemm_tc_kernel", full),
                                 "flops": wo_flops(wl)}})
    del d, bufs, step
    return out


def setup_workload(name, torch):
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import pipeline as P
    wl = W.WORKLOADS[name]
    if wl.kind == "append":
        return setup_append(wl, torch)
    x = W.make_inputs(wl)

    def dev(a):
        return torch.from_numpy(W.to_bf16(a)[1]).view(torch.bfloat16).cuda()

    d = {"q_nope": dev(x.q_nope), "q_pe": dev(x.q_pe), "wk_b": dev(x.wk_b), "wv_b": dev(x.wv_b)}
    kv = torch.from_numpy(x.kv_rows_bits()).view(torch.bfloat16).cuda()
    if wl.cache == "q8_0":
        n = kv.shape[0]
        d["kv_q"] = torch.empty(n, 576, dtype=torch.int8, device="cuda")
        d["kv_d"] = torch.empty(18, n, dtype=torch.float16, device="cuda")
        mla.mla_quantize_q8_0(kv, d["kv_q"], d["kv_d"])         # the cache producer, outside the timing
        del kv
    else:
        d["kv"] = kv
    if wl.kind == "decode":
        d["seq_start"] = torch.from_numpy(x.seq_start).cuda()
        d["seq_len"] = torch.from_numpy(x.seq_len).cuda()
        max_len = int(x.seq_len.max())
        bufs = P.decode_buffers(wl.B, wl.n_head, max_len)

        def step(stream=None, ev=None):
            mla.mla_absorb_q(d["q_nope"], d["wk_b"], bufs.q_lat, stream=stream)
            if ev:
                ev[0].record()
            if wl.cache == "q8_0":
                mla.mla_attn_decode_q8_0(bufs.q_lat, d["q_pe"], d["kv_q"], d["kv_d"], d["seq_start"], d["seq_len"],
                                         max_len, bufs.workspace, bufs.o_lat, stream=stream)
            else:
                mla.mla_attn_decode(bufs.q_lat, d["q_pe"], d["kv"], d["seq_start"], d["seq_len"], max_len,
                                    bufs.workspace, bufs.o_lat, stream=stream)
            if ev:
                ev[1].record()
            mla.mla_late_decompress(bufs.o_lat, d["wv_b"], bufs.o, stream=stream)
        launches = 4
    else:
        bufs = P.prefill_buffers(wl.T, wl.n_head, n_kv=x.n_rows)

        def step(stream=None, ev=None):
            mla.mla_absorb_q(d["q_nope"], d["wk_b"], bufs.q_lat, stream=stream)
            if ev:
                ev[0].record()
            if wl.cache == "q8_0":
                mla.mla_attn_prefill_q8_0(bufs.q_lat, d["q_pe"], d["kv_q"], d["kv_d"], wl.q_pos0, bufs.o_lat,
                                          stream=stream, workspace=bufs.workspace)
            else:
                mla.mla_attn_prefill(bufs.q_lat, d["q_pe"], d["kv"], wl.q_pos0, bufs.o_lat, stream=stream,
                                     workspace=bufs.workspace)
            if ev:
                ev[1].record()
            mla.mla_late_decompress(bufs.o_lat, d["wv_b"], bufs.o, stream=stream)
        launches = 4    # absorb, fp16 cache staging, attention, late decompression
    return wl, x, d, bufs, step, launches


def time_steps(torch, step, steps, warmup, flush):
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    step_ms, attn_ms = [], []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step(ev=(a0, a1))
        e1.record()
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        attn_ms.append(a0.elapsed_time(a1))
    return step_ms, attn_ms


def max_over_ranks(value: float, torch, dist, device: str) -> float:
    """The slowest rank's value (N replicas: the job ends when the last one
    does); the value itself without a process group."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_of(wl, x, attn_ms, pk, pk_kind):
    """Roofline of the step's dominant kernel (the attention kernel, with the
    decode combine; the append kernel) from its measured average duration."""
    if wl.kind == "prefill":
        ach = attn_flops(wl, x) / (attn_ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(ach, 3), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "peak_kind": f"{pk_kind} bf16 dense, burst"}
        if "bf16_tflops_sustained" in pk:
            roof["frac_of_sustained"] = round(ach / pk["bf16_tflops_sustained"], 4)
    else:
        units = append_bytes(wl) if wl.kind == "append" else decode_bytes(wl, x)
        ach = units / (attn_ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_kind": f"{pk_kind} HBM copy"}
        if wl.kind == "decode":
            tf = attn_flops(wl, x) / (attn_ms * 1e-3) / 1e12
            roof["tensor_tflops"] = round(tf, 2)
            roof["tensor_frac"] = round(tf / pk["bf16_tflops"], 4)
    kname = "rope_append_kernel" if wl.kind == "append" else "attn_tc_kernel"
    roof["traffic"] = recorded_traffic(kname, wl.name)
    roof["kernel"] = kname if wl.kind != "decode" else "attn_tc_kernel+combine_kernel"
    roof["attn_ms"] = round(attn_ms, 4)
    return roof


def measure(args, torch, name, flush, pk, pk_kind, world=1, with_e2e=True):
    """Time `steps` whole steps of one workload (after `warmup` untimed ones),
    L2 flushed before each; returns the per-workload figures, the live inputs
    and the raw per-step times."""
    wl, x, d, bufs, step, launches = setup_workload(name, torch)
    torch.cuda.synchronize()
    step_ms, attn_ms = time_steps(torch, step, args.steps, args.warmup, flush)
    ms = sum(step_ms) / len(step_ms)
    attn = sum(attn_ms) / len(attn_ms)
    if wl.kind == "prefill":
        value, unit = attn_flops(wl, x) * world / (ms * 1e-3) / 1e12, "TFLOP/s"
    else:
        units = append_bytes(wl) if wl.kind == "append" else decode_bytes(wl, x)
        value, unit = units * world / (ms * 1e-3) / 1e9, "GB/s"
    out = {"workload": wl.name, "value": round(value, 3), "unit": unit, "ms_per_step": round(ms, 4),
           "roofline": roofline_of(wl, x, attn, pk, pk_kind), "gpu_launches": launches * args.steps}
    if wl.kind == "prefill":
        out["tokens_per_s"] = round(wl.T / (ms * 1e-3), 1)
    elif wl.kind == "decode":
        out["tokens_per_s"] = round(wl.B / (ms * 1e-3), 1)
    if with_e2e:
        if wl.kind == "prefill":
            out["e2e"] = e2e_prefill(args, torch, wl, x, d, bufs)
        elif wl.kind == "append":
            out["e2e"] = e2e_append(args, torch, wl, d, bufs)
        else:
            out["e2e"] = e2e_decode(args, torch, wl, x, d, bufs)
    return out, (wl, x), sum(step_ms)


def run_ours(args, torch, dist, rank, world):
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import build
    if rank == 0 or not os.path.exists(build.LIB):
        build.build()
    if dist is not None:
        dist.barrier()
    mla.load_library()
    pk, pk_kind = peaks()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")

    if ":" in args.workload:              # a materialised or projected prefill as the headline
        out = measure_variant(args, torch, args.workload, flush, pk, pk_kind, world)
        out.update({"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                    "data": "synthetic", "config": {"workload": args.workload}})
        return out
    # the headline workload: clocks sampled during its timed steps
    wl, x, d, bufs, step, launches = setup_workload(args.workload, torch)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_wall = time.perf_counter()
        step_ms, attn_ms = time_steps(torch, step, args.steps, args.warmup, flush)
        t_wall = time.perf_counter() - t_wall
    err = mla.mla_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error {err} during the bench")
    total_ms = max_over_ranks(sum(step_ms), torch, dist, "cuda")
    ms_step = total_ms / args.steps
    attn_avg = sum(attn_ms) / len(attn_ms)
    if wl.kind == "prefill":
        value, unit = attn_flops(wl, x) * world / (ms_step * 1e-3) / 1e12, "TFLOP/s"
    else:
        units = append_bytes(wl) if wl.kind == "append" else decode_bytes(wl, x)
        value, unit = units * world / (ms_step * 1e-3) / 1e9, "GB/s"

    out = {"metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.cache == "bf16" else "bf16+q8_0 cache",
           "data": "synthetic (seeded N(0,1) activations, N(0,1/sqrt(fan_in)) weights)",
           "config": {"workload": wl.name, "describe": wl.describe, "n_head": wl.n_head, "cache": wl.cache,
                      "T": wl.T, "q_pos0": wl.q_pos0, "n_kv": wl.n_kv, "B": wl.B,
                      "parallelism": "replicas" if world > 1 else "single GPU",
                      "l2": "flushed before every step (512 MB write)"},
           "roofline": roofline_of(wl, x, attn_avg, pk, pk_kind), "gpu_launches": launches * args.steps,
           "clocks": clk.summary(), "wall_s_timed": round(t_wall, 3)}
    if wl.kind == "prefill":
        out["tokens_per_s"] = round(wl.T * world / (ms_step * 1e-3), 1)
        out["e2e"] = e2e_prefill(args, torch, wl, x, d, bufs)
    elif wl.kind == "append":
        out["e2e"] = e2e_append(args, torch, wl, d, bufs)
    else:
        out["e2e"] = e2e_decode(args, torch, wl, x, d, bufs)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, x, unit, budget_s=args.cpu_budget)
    del d, bufs, step
    torch.cuda.empty_cache()

    # every other workload, one after the other (replicas: each rank its own)
    names = [n for n in secondary_names(args) if n != wl.name]
    if names:
        out["secondary"] = {}
        for name in names:
            if ":" in name:
                sec = measure_variant(args, torch, name, flush, pk, pk_kind, world)
            else:
                sec, (swl, sx), _ = measure(args, torch, name, flush, pk, pk_kind, world)
                if rank == 0 and world == 1 and not args.no_cpu_baseline:
                    # a smaller sample than the headline's; decode on 16 heads
                    sec["cpu_baseline"] = cpu_baseline(swl, sx, sec["unit"], budget_s=args.cpu_budget / 4,
                                                       n_heads=16 if swl.kind == "decode" else None)
            if mla.mla_get_device_error() != 0:
                raise RuntimeError(f"device error during the {name} bench")
            out["secondary"][name] = sec
            out["gpu_launches"] += sec["gpu_launches"]
            torch.cuda.empty_cache()
    return out


def secondary_names(args):
    if args.secondary == "none":
        return []
    if args.secondary == "all":
        return list(SECONDARY_WORKLOADS)
    names = [n for n in args.secondary.split(",") if n]
    for n in names:
        base, _, variant = n.partition(":")
        if base not in W.WORKLOADS or variant not in ("", "materialized", "projected"):
            raise SystemExit(f"unknown workload {n}")
    return names


def e2e_overlapped(args, torch, d, out, step):
    """The step through the public entry points with pinned host buffers: every
    step copies all its inputs host->device and its output device->host, on a
    copy stream that overlaps them with the neighbouring steps' compute
    (pipeline.HostOverlap).  Returns (ms per step, h2d bytes, d2h bytes)."""
    from mla_latent_kv_lat_gb300 import pipeline as P
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    dev = [d, {k: torch.empty_like(v) for k, v in d.items()}]
    outs = [out, torch.empty_like(out)]
    run = P.HostOverlap(host, dev, outs, step)
    run.run(args.warmup)
    ms = run.run(args.steps) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    del dev, outs, run
    return ms, h2d, d2h


def e2e_prefill(args, torch, wl, x, d, bufs):
    """Same metric through the public pipeline with pinned host buffers: every
    step copies its inputs host->device and the output o device->host (copies
    overlapped with the neighbouring steps' compute)."""
    from mla_latent_kv_lat_gb300 import pipeline as P

    def step(dv, out):
        P.mla_prefill(dv["q_nope"], dv["q_pe"], dv["wk_b"], dv["wv_b"], wl.q_pos0, kv=dv.get("kv"),
                      kv_q=dv.get("kv_q"), kv_d=dv.get("kv_d"), bufs=P.PrefillBuffers(bufs.q_lat, bufs.o_lat, out,
                                                                                      None, bufs.workspace))
    ms, h2d, d2h = e2e_overlapped(args, torch, d, bufs.o, step)
    return {"value": round(attn_flops(wl, x) / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "overlapped with the neighbouring steps (copy stream, two buffer sets)"}


def e2e_append(args, torch, wl, d, caches):
    """The append through the public entry point with its inputs copied from
    pinned host memory every step; the step's result is the cache rows in HBM
    (read by the attention kernels there), so the host reads back only the
    device status word that says they were all written."""
    import mla_latent_kv_lat_gb300 as mla
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())

    def one():
        for k, t in host.items():
            d[k].copy_(t, non_blocking=True)
        mla.mla_rope_append(d["c_kv"], d["k_pe"], d["pos"], d["slot"], **caches)
        if mla.mla_get_device_error() != 0:
            raise RuntimeError("device error during the append e2e run")

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        one()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = sum(ts) / len(ts)
    return {"value": round(append_bytes(wl) / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4}


def e2e_decode(args, torch, wl, x, d, bufs):
    """The decode step with every input, the cache included, copied from pinned
    host memory each step and o read back (copies overlapped as for prefill)."""
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import pipeline as P
    max_len = int(x.seq_len.max())

    def step(dv, out):
        kw = dict(kv_q=dv["kv_q"], kv_d=dv["kv_d"]) if wl.cache == "q8_0" else dict(kv=dv["kv"])
        mla.mla_decode(dv["q_nope"], dv["q_pe"], dv["wk_b"], dv["wv_b"], dv["seq_start"], dv["seq_len"], max_len,
                       bufs=P.DecodeBuffers(bufs.q_lat, bufs.o_lat, out, bufs.workspace), **kw)
    ms, h2d, d2h = e2e_overlapped(args, torch, d, bufs.o, step)
    return {"value": round(decode_bytes(wl, x) / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "overlapped with the neighbouring steps (copy stream, two buffer sets)"}


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(wl: W.Workload, x, rows: int, n_heads=None):
    """Run the oracle (un-absorbed definition) on the first `rows` query rows
    (prefill), sequences (decode) or new tokens (append); returns (seconds,
    units done).  Decode with `n_heads`: only heads [0, n_heads), the seconds
    scaled by n_head / n_heads (the oracle's work is proportional to heads)."""
    from oracle import mla_oracle as O
    t0 = time.perf_counter()
    if wl.kind == "append":
        r = O.cache_rows(x.c_kv[:rows], x.k_pe[:rows], x.pos[:rows], 10000.0, 0.025)
        O.quantize_q8_0(r.astype(np.float32))
        return time.perf_counter() - t0, rows * APPEND_TOKEN_BYTES
    if wl.kind == "prefill":
        c_kv, k_pe = x.c_kv, x.k_pe
        if wl.cache == "q8_0":
            codes, scales = O.quantize_q8_0(np.concatenate([c_kv, k_pe], axis=1))
            deq = O.dequantize_q8_0(codes, scales)
            c_kv, k_pe = deq[:, :512], deq[:, 512:]
            t0 = time.perf_counter()
        sel = np.arange(wl.T - rows, wl.T)          # the last rows see the most keys
        O.attention_unabsorbed(x.q_nope[sel], x.q_pe[sel], c_kv, k_pe, x.wk_b, x.wv_b, x.q_pos()[sel], wl.scale)
        pairs = int((x.q_pos()[sel] + 1).sum())
        units = pairs * wl.n_head * FLOP_PER_PAIR_HEAD
    else:
        seqs = list(range(rows))
        heads = None if n_heads is None else list(range(n_heads))
        O.decode_unabsorbed(x.q_nope, x.q_pe, x.c_kv, x.k_pe, x.wk_b, x.wv_b, x.seq_start, x.seq_len, wl.scale,
                            heads=heads, seqs=seqs)
        row = 576 * 2 if wl.cache == "bf16" else 612
        units = int(x.seq_len[seqs].astype(np.int64).sum()) * row + len(seqs) * wl.n_head * (576 + 512) * 2
        if n_heads is not None:
            return (time.perf_counter() - t0) * wl.n_head / n_heads, units
    return time.perf_counter() - t0, units


def cpu_baseline(wl, x, unit, budget_s=20.0, n_heads=None):
    rows = 4 if wl.kind != "decode" else 1
    cap = wl.B if wl.kind == "decode" else wl.T
    sec, units = oracle_sample(wl, x, rows, n_heads)
    # grow the sample toward the time budget, then report the largest
    while sec < budget_s / 4 and rows < cap:
        rows = min(rows * 4, cap)
        sec, units = oracle_sample(wl, x, rows, n_heads)
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    heads = "all heads" if n_heads is None else f"heads 0-{n_heads - 1} of {wl.n_head}, time scaled to all"
    what = {"prefill": f"last {rows} query rows (all heads)", "decode": f"first {rows} sequences ({heads})",
            "append": f"first {rows} new tokens (rows + q8_0)"}[wl.kind]
    return {"value": units / sec / scale, "unit": unit, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{what} of {wl.name}, un-absorbed numpy fp64 oracle, {sec:.2f} s"}


def run_reference(args):
    wl = W.WORKLOADS[args.workload]
    x = W.make_append_inputs(wl.T, wl.n_kv) if wl.kind == "append" else W.make_inputs(wl)
    unit = "TFLOP/s" if wl.kind == "prefill" else "GB/s"
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    rows = {"prefill": 32, "decode": 1, "append": 4096}[wl.kind]
    for _ in range(args.warmup):
        oracle_sample(wl, x, rows)
    tot_s = tot_u = 0.0
    for _ in range(args.steps):
        s, u = oracle_sample(wl, x, rows)
        tot_s += s
        tot_u += u
    value = tot_u / tot_s / scale
    what = {"prefill": f"last {rows} query rows", "decode": f"first {rows} sequence",
            "append": f"first {rows} new tokens"}[wl.kind]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "describe": wl.describe},
            "cpu_baseline": {"value": value, "unit": unit, "cores": blas_threads(), "kind": "oracle",
                             "sample": f"{what} of {wl.name} per step"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def sweep_decode(args, torch):
    """Decode attention (+ combine) of 32 sequences x 128 heads at a range of
    cache lengths, bf16 and q8_0 cache (the llama-sweep-bench way of reading
    a decode kernel: throughput against N_KV).  Seeded device-side N(0,1)
    inputs; one JSON line per point.  Not part of the default bench line."""
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import build
    from mla_latent_kv_lat_gb300 import pipeline as P
    build.build()
    mla.load_library()
    pk, pk_kind = peaks()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)
    B, H = 32, 128
    out = []
    for L in (1024, 4096, 16384, 32768, 65536):
        n = B * L
        kv = torch.randn(n, 576, device="cuda", generator=g).to(torch.bfloat16)
        kv_q = torch.empty(n, 576, dtype=torch.int8, device="cuda")
        kv_d = torch.empty(18, n, dtype=torch.float16, device="cuda")
        mla.mla_quantize_q8_0(kv, kv_q, kv_d)
        q_lat = torch.randn(B, H, 512, device="cuda", generator=g).to(torch.float16)
        q_pe = torch.randn(B, H, 64, device="cuda", generator=g).to(torch.bfloat16)
        seq_len = torch.full((B,), L, dtype=torch.int32, device="cuda")
        seq_start = torch.arange(B, dtype=torch.int64, device="cuda") * L
        bufs = P.decode_buffers(B, H, L)
        for cache, row in (("bf16", 1152), ("q8_0", 612)):
            def step(stream=None, ev=None):
                if ev:
                    ev[0].record()
                if cache == "bf16":
                    mla.mla_attn_decode(q_lat, q_pe, kv, seq_start, seq_len, L, bufs.workspace, bufs.o_lat)
                else:
                    mla.mla_attn_decode_q8_0(q_lat, q_pe, kv_q, kv_d, seq_start, seq_len, L, bufs.workspace,
                                             bufs.o_lat)
                if ev:
                    ev[1].record()
            _, attn_ms = time_steps(torch, step, args.steps, args.warmup, flush)
            ms = sorted(attn_ms)[len(attn_ms) // 2]
            nbytes = n * row + B * H * (576 + 512) * 2
            gbs = nbytes / (ms * 1e-3) / 1e9
            out.append({"sweep": "decode", "cache": cache, "B": B, "n_head": H, "cache_len": L,
                        "ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                        "TFLOP/s": round(n * H * FLOP_PER_PAIR_HEAD / (ms * 1e-3) / 1e12, 1)})
        if mla.mla_get_device_error() != 0:
            raise RuntimeError("device error during the decode sweep")
        del kv, kv_q, kv_d
    return out


def sweep_prefill(args, torch):
    """Prefill attention (staging included) against chunk length: the Lite
    shape (16 heads) causal over its own cache, and the V3 shape (128 heads)
    at position 32768 over a cache ending with the chunk.  Seeded device-side
    N(0,1) inputs; one JSON line per point.  Not part of the default line."""
    import mla_latent_kv_lat_gb300 as mla
    from mla_latent_kv_lat_gb300 import build
    build.build()
    mla.load_library()
    pk, pk_kind = peaks()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)
    out = []
    points = [(16, T, 0) for T in (1024, 2048, 4096, 8192, 16384)] + [(128, T, 32768) for T in (512, 1024, 2048, 4096)]
    for H, T, q_pos0 in points:
        n_kv = q_pos0 + T
        kv = torch.randn(n_kv, 576, device="cuda", generator=g).to(torch.bfloat16)
        q_lat = torch.randn(T, H, 512, device="cuda", generator=g).to(torch.float16)
        q_pe = torch.randn(T, H, 64, device="cuda", generator=g).to(torch.bfloat16)
        o_lat = torch.empty(T, H, 512, dtype=torch.float16, device="cuda")
        ws = torch.empty(mla.mla_prefill_workspace_size(H, n_kv), dtype=torch.uint8, device="cuda")

        def step(stream=None, ev=None):
            if ev:
                ev[0].record()
            mla.mla_attn_prefill(q_lat, q_pe, kv, q_pos0, o_lat, workspace=ws)
            if ev:
                ev[1].record()
        _, attn_ms = time_steps(torch, step, args.steps, args.warmup, flush)
        ms = sorted(attn_ms)[len(attn_ms) // 2]
        flops = float(T * q_pos0 + T * (T + 1) // 2) * H * FLOP_PER_PAIR_HEAD
        tf = flops / (ms * 1e-3) / 1e12
        out.append({"sweep": "prefill", "n_head": H, "T": T, "q_pos0": q_pos0, "row_tiles": (T * H + 127) // 128,
                    "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / pk["bf16_tflops"], 4)})
        if mla.mla_get_device_error() != 0:
            raise RuntimeError("device error during the prefill sweep")
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="headline workload: one of " + ", ".join(sorted(W.WORKLOADS)) +
                         " (a prefill may take :materialized or :projected)")
    ap.add_argument("--chunk", type=int, default=0,
                    help="prefill: time the last CHUNK queries of the workload instead of all of them (same "
                         "shape and positions; for small profiling cases)")
    ap.add_argument("--secondary", default="all",
                    help="workloads measured after the headline one: all (default), none, or a comma list")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-decode", action="store_true",
                    help="instead of the bench line: decode throughput against cache length (one JSON line each)")
    ap.add_argument("--sweep-prefill", action="store_true",
                    help="instead of the bench line: prefill throughput against chunk length (one JSON line each)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    base, _, variant = args.workload.partition(":")
    if base not in W.WORKLOADS or variant not in ("", "materialized", "projected"):
        raise SystemExit(f"unknown workload {args.workload}")
    if args.chunk:
        wl = W.WORKLOADS[base]
        if wl.kind != "prefill" or not 0 < args.chunk <= wl.T:
            raise SystemExit("--chunk applies to prefill workloads, 0 < CHUNK <= T")
        # the last CHUNK queries: positions q_pos0 + T - CHUNK .., over the same cache
        import dataclasses
        W.WORKLOADS[base] = dataclasses.replace(wl, name=f"{base}_last{args.chunk}", T=args.chunk,
                                                q_pos0=wl.q_pos0 + wl.T - args.chunk)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if args.sweep_decode or args.sweep_prefill:
        for row in (sweep_decode if args.sweep_decode else sweep_prefill)(args, torch):
            print(json.dumps(row), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    out = run_ours(args, torch, dist, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
