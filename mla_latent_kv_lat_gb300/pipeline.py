"""The whole absorbed-MLA hot path as one call per use case.

Prefill: absorb (wk_b into the query) -> causal latent attention -> late
decompression (wv_b).  Decode: the same with split-KV attention.  Each step is
one C-ABI call of libmla on the caller's stream; this module only allocates
the intermediate device buffers through PyTorch and, for the host variants,
moves inputs and outputs between pinned host memory and the device.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import binding as B


@dataclass
class PrefillBuffers:
    q_lat: torch.Tensor      # fp16 [T, H, 512]
    o_lat: torch.Tensor      # fp16 [T, H, 512]
    o: torch.Tensor          # fp32 [T, H, 128]
    lse: Optional[torch.Tensor] = None
    workspace: Optional[torch.Tensor] = None   # uint8, >= mla_prefill_workspace_size(H, n_kv)


def prefill_buffers(T: int, H: int, device="cuda", with_lse=False, n_kv: Optional[int] = None) -> PrefillBuffers:
    """Device buffers of one prefill; with ``n_kv`` also the attention
    workspace for a cache of that many rows (else each call allocates it)."""
    ws = None
    if n_kv is not None:
        ws = torch.empty(B.mla_prefill_workspace_size(H, n_kv), dtype=torch.uint8, device=device)
    return PrefillBuffers(
        torch.empty(T, H, B.KV_LORA_RANK, dtype=torch.float16, device=device),
        torch.empty(T, H, B.KV_LORA_RANK, dtype=torch.float16, device=device),
        torch.empty(T, H, B.V_HEAD, dtype=torch.float32, device=device),
        torch.empty(T, H, dtype=torch.float32, device=device) if with_lse else None, ws)


def mla_prefill(q_nope, q_pe, wk_b, wv_b, q_pos0: int, *, kv=None, kv_q=None, kv_d=None,
                bufs: Optional[PrefillBuffers] = None, scale=None, stream=None) -> PrefillBuffers:
    """o = late_decompress(attn(absorb(q_nope), q_pe, cache)) on device tensors.

    Pass ``kv`` (bf16 [n_kv, 576]) or ``kv_q``/``kv_d`` (q8_0 cache)."""
    T, H = q_nope.shape[0], q_nope.shape[1]
    if bufs is None:
        bufs = prefill_buffers(T, H, q_nope.device, n_kv=(kv if kv is not None else kv_q).shape[0])
    B.mla_absorb_q(q_nope, wk_b, bufs.q_lat, scale=scale, stream=stream)
    if kv is not None:
        B.mla_attn_prefill(bufs.q_lat, q_pe, kv, q_pos0, bufs.o_lat, bufs.lse, scale=scale, stream=stream,
                           workspace=bufs.workspace)
    else:
        B.mla_attn_prefill_q8_0(bufs.q_lat, q_pe, kv_q, kv_d, q_pos0, bufs.o_lat, bufs.lse, scale=scale,
                                stream=stream, workspace=bufs.workspace)
    B.mla_late_decompress(bufs.o_lat, wv_b, bufs.o, scale=scale, stream=stream)
    return bufs


@dataclass
class ProjectBuffers:
    o16: torch.Tensor        # fp16 [T, H, 128]: late decompression's output for the projection
    u: torch.Tensor          # fp32 [T, D]


def project_buffers(T: int, H: int, D: int, device="cuda") -> ProjectBuffers:
    return ProjectBuffers(torch.empty(T, H, B.V_HEAD, dtype=torch.float16, device=device),
                          torch.empty(T, D, dtype=torch.float32, device=device))


def mla_prefill_projected(q_nope, q_pe, wk_b, wv_b, w_o, q_pos0: int, *, kv=None, kv_q=None, kv_d=None,
                          bufs: Optional[PrefillBuffers] = None, pbufs: Optional[ProjectBuffers] = None,
                          scale=None, stream=None):
    """The path followed by the output projection: absorb -> latent attention ->
    late decompression (fp16 o) -> u = o . w_o, with w_o the fp16 weight
    (mla_convert_bf16_to_f16 of the model's bf16 w_o, once).  Returns (bufs, pbufs)."""
    T, H = q_nope.shape[0], q_nope.shape[1]
    if bufs is None:
        bufs = prefill_buffers(T, H, q_nope.device, n_kv=(kv if kv is not None else kv_q).shape[0])
    if pbufs is None:
        pbufs = project_buffers(T, H, w_o.shape[2], q_nope.device)
    B.mla_absorb_q(q_nope, wk_b, bufs.q_lat, scale=scale, stream=stream)
    if kv is not None:
        B.mla_attn_prefill(bufs.q_lat, q_pe, kv, q_pos0, bufs.o_lat, bufs.lse, scale=scale, stream=stream,
                           workspace=bufs.workspace)
    else:
        B.mla_attn_prefill_q8_0(bufs.q_lat, q_pe, kv_q, kv_d, q_pos0, bufs.o_lat, bufs.lse, scale=scale,
                                stream=stream, workspace=bufs.workspace)
    B.mla_late_decompress_f16(bufs.o_lat, wv_b, pbufs.o16, scale=scale, stream=stream)
    B.mla_output_project(pbufs.o16, w_o, pbufs.u, scale=scale, stream=stream)
    return bufs, pbufs


@dataclass
class DecodeBuffers:
    q_lat: torch.Tensor
    o_lat: torch.Tensor
    o: torch.Tensor
    workspace: torch.Tensor


def decode_buffers(Bn: int, H: int, max_len: int, device="cuda") -> DecodeBuffers:
    ws = B.mla_decode_workspace_size(H, Bn, max_len)
    return DecodeBuffers(
        torch.empty(Bn, H, B.KV_LORA_RANK, dtype=torch.float16, device=device),
        torch.empty(Bn, H, B.KV_LORA_RANK, dtype=torch.float16, device=device),
        torch.empty(Bn, H, B.V_HEAD, dtype=torch.float32, device=device),
        torch.empty(ws, dtype=torch.uint8, device=device))


def mla_decode(q_nope, q_pe, wk_b, wv_b, seq_start, seq_len, max_len: int, *, kv=None, kv_q=None, kv_d=None,
               bufs: Optional[DecodeBuffers] = None, scale=None, stream=None) -> DecodeBuffers:
    """One decode step for B sequences (one new token each) on device tensors."""
    Bn, H = q_nope.shape[0], q_nope.shape[1]
    if bufs is None:
        bufs = decode_buffers(Bn, H, max_len, q_nope.device)
    B.mla_absorb_q(q_nope, wk_b, bufs.q_lat, scale=scale, stream=stream)
    if kv is not None:
        B.mla_attn_decode(bufs.q_lat, q_pe, kv, seq_start, seq_len, max_len, bufs.workspace, bufs.o_lat,
                          scale=scale, stream=stream)
    else:
        B.mla_attn_decode_q8_0(bufs.q_lat, q_pe, kv_q, kv_d, seq_start, seq_len, max_len, bufs.workspace,
                               bufs.o_lat, scale=scale, stream=stream)
    B.mla_late_decompress(bufs.o_lat, wv_b, bufs.o, scale=scale, stream=stream)
    return bufs


def mla_prefill_host(host: dict, q_pos0: int, dev: dict, bufs: PrefillBuffers, out_host: torch.Tensor,
                     stream=None) -> torch.Tensor:
    """Host-buffer prefill: copy each pinned host input into its device buffer,
    run the path, copy o back into pinned ``out_host``.  ``host``/``dev`` map
    input names (q_nope, q_pe, wk_b, wv_b and kv or kv_q/kv_d) to tensors."""
    for k, t in host.items():
        dev[k].copy_(t, non_blocking=True)
    mla_prefill(dev["q_nope"], dev["q_pe"], dev["wk_b"], dev["wv_b"], q_pos0, kv=dev.get("kv"),
                kv_q=dev.get("kv_q"), kv_d=dev.get("kv_d"), bufs=bufs, stream=stream)
    out_host.copy_(bufs.o, non_blocking=True)
    return out_host


class HostOverlap:
    """Steps of the path on pinned host buffers, with the copies overlapped.

    Every step copies its inputs host -> device and its output device -> host,
    but on a copy stream of their own: step k+1's inputs go in and step k-1's
    output comes out while step k computes on the compute stream.  Two device
    input sets and two device outputs alternate; events order each copy
    against the steps that use its buffers.  ``step(dev, out)`` enqueues one
    step's kernels on the current stream, reading the input tensors in the
    dict ``dev`` and writing ``out``.
    """

    def __init__(self, host: dict, dev_sets, outs, step):
        self.host = host
        self.dev = dev_sets                     # two dicts of device inputs (same keys as host)
        self.outs = outs                        # two device outputs
        self.step = step
        self.host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
        self.copy = torch.cuda.Stream()
        self.compute = torch.cuda.Stream()

    def run(self, n: int) -> float:
        """Run n steps; return the milliseconds from the first copy in to the
        last copy out (CUDA events)."""
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()

        def copy_in(k):
            s = k % 2
            with torch.cuda.stream(self.copy):
                if k >= 2:
                    self.copy.wait_event(ev_done[s])      # step k-2 no longer reads this input set
                for key, t in self.host.items():
                    self.dev[s][key].copy_(t, non_blocking=True)
                ev_in[s].record(self.copy)

        t0.record(self.copy)
        copy_in(0)
        for k in range(n):
            s = k % 2
            with torch.cuda.stream(self.compute):
                self.compute.wait_event(ev_in[s])
                self.step(self.dev[s], self.outs[s])
                ev_done[s].record(self.compute)
            if k + 1 < n:
                copy_in(k + 1)
            with torch.cuda.stream(self.copy):
                self.copy.wait_event(ev_done[s])
                self.host_out[s].copy_(self.outs[s], non_blocking=True)
        t1.record(self.copy)
        t1.synchronize()
        return t0.elapsed_time(t1)
