"""Run a described fusion (transpose_heroes_gb300.inputs.Fusion) through the C ABI on device buffers.

DeviceFusion holds the device copies of a fusion's operands and its output buffer; run() enqueues the
fusion on a stream with one C-ABI call. Host<->device copies use pinned staging buffers so that they
can be asynchronous and timed end to end.
"""

from __future__ import annotations

import numpy as np
import torch

from . import (layout_convert, quant_binary, quant_fusion, reduce_fusion, reduce_max_argmax, reduce_workspace_size,
               transpose_fusion)
from .inputs import ELEM_BYTES, Fusion

# physical buffers as torch tensors of the same element size (16-bit floats carried as int16 bits)
_TORCH = {"f32": torch.float32, "bf16": torch.int16, "f16": torch.int16, "s8": torch.int8, "s32": torch.int32}
_NP = {"f32": np.float32, "bf16": np.int16, "f16": np.int16, "s8": np.int8, "s32": np.int32}
_NP_OUT = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "s8": np.int8, "s32": np.int32}


def host_tensor(arr: np.ndarray, dtype: str, pin: bool = False) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr).view(_NP[dtype]))
    return t.pin_memory() if pin else t


def _numel(dims) -> int:
    return int(np.prod(dims)) if len(dims) else 1


class DeviceFusion:
    """Device-resident operands and output of one fusion instance."""

    def __init__(self, f: Fusion, device="cuda", pin_host: bool = False):
        self.f = f
        self.device = device
        self.host_in = host_tensor(f.data, f.dtype, pin=pin_host)
        self.x = self.host_in.to(device)
        self.bcast = None
        self.host_bcast = None
        for chain in (f.prologue, f.epilogue):
            if chain and chain.get("bcast") is not None:
                b = chain["bcast"]
                self.host_bcast = host_tensor(b["data"], b["dtype"], pin=pin_host)
                self.bcast = self.host_bcast.to(device)
        self.qin = self.qout = None
        if f.in_q is not None:
            self.qin = self._quant(f.in_q)
        if f.out_q is not None:
            self.qout = self._quant(f.out_q)
        n_out = _numel(f.out_dims) if f.out_dims is not None else 1
        self.out = torch.empty(n_out, dtype=_TORCH[f.out_dtype], device=device)
        self.host_out = torch.empty(n_out, dtype=_TORCH[f.out_dtype], pin_memory=pin_host)
        self.out_idx = torch.empty(n_out, dtype=torch.int32, device=device) if f.kind == "argmax" else None
        # the reduce's scratch (row partials when few long rows are split), allocated once
        self.workspace = None
        if f.kind == "reduce":
            nbytes = reduce_workspace_size(f.dims, f.dtype, f.dimensions, in_m2m=f.m2m)
            if nbytes:
                self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.rhs = None
        if f.kind == "quant_binary":
            self.rhs = host_tensor(f.rhs, f.dtype).to(device)
            self._qspec = lambda q: {"host_scales": q["scales"], "host_zero_points": q["zero_points"],
                                     "quantization_dimension": None, "storage_min": q.get("storage_min", -128),
                                     "storage_max": q.get("storage_max", 127)}

    def _quant(self, q):
        scales = np.ascontiguousarray(np.atleast_1d(q["scales"]), dtype=np.float32)
        zps = np.ascontiguousarray(np.atleast_1d(q["zero_points"]), dtype=np.int32)
        return {"scales": torch.from_numpy(scales).to(self.device), "zero_points": torch.from_numpy(zps).to(self.device),
                "host_scales": scales, "host_zero_points": zps, "quantization_dimension": q.get("quantization_dimension"),
                "storage_min": q.get("storage_min", -128), "storage_max": q.get("storage_max", 127)}

    def _chain(self, spec):
        if spec is None:
            return None
        spec = dict(spec)
        if spec.get("bcast") is not None:
            b = dict(spec["bcast"])
            b["tensor"] = self.bcast
            spec["bcast"] = b
        return spec

    def run(self, stream=None):
        f = self.f
        if f.kind == "reduce":
            ws = self.workspace
            reduce_fusion(self.x, f.dims, f.dtype, f.dimensions, f.reduce_kind, f.init, self.out, f.out_dtype,
                          in_m2m=f.m2m, out_m2m=f.out_m2m, prologue=self._chain(f.prologue), workspace=ws,
                          workspace_bytes=0 if ws is None else ws.numel(), stream=stream)
        elif f.kind == "transpose":
            transpose_fusion(self.x, f.dims, f.dtype, f.permutation, self.out, in_m2m=f.m2m, out_m2m=f.out_m2m,
                             prologue=self._chain(f.prologue), self_add=f.self_add,
                             epilogue=self._chain(f.epilogue), stream=stream)
        elif f.kind == "layout":
            layout_convert(self.x, f.dims, f.dtype, f.m2m, f.out_m2m, self.out, stream=stream)
        elif f.kind == "quant":
            quant_fusion(self.x, f.dims, self.qin, f.out_m2m, self.out, out_dtype=f.out_dtype, out_q=self.qout,
                         in_m2m=f.m2m, float_ops=self._chain(f.prologue), stream=stream)
        elif f.kind == "quant_binary":
            quant_binary(f.op, self.x, self.rhs, f.dims, self._qspec(f.in_q), self._qspec(f.in_q), self.out,
                         self._qspec(f.out_q), lhs_m2m=f.m2m, rhs_m2m=f.m2m, out_m2m=f.out_m2m, stream=stream)
        elif f.kind == "argmax":
            reduce_max_argmax(self.x, f.dims, f.dtype, f.dimensions, self.out, self.out_idx, init_value=f.init,
                              init_index=-1, in_m2m=f.m2m, out_m2m=f.out_m2m, out_idx_m2m=f.out_m2m, stream=stream)
        else:
            raise ValueError(f"unknown fusion kind {f.kind}")
        return self.out

    # end-to-end step: host input -> device, fusion, device output -> host (all on `stream`)
    def h2d(self, stream=None):
        self.x.copy_(self.host_in, non_blocking=True)
        if self.bcast is not None:
            self.bcast.copy_(self.host_bcast, non_blocking=True)

    def d2h(self):
        self.host_out.copy_(self.out, non_blocking=True)

    @property
    def h2d_bytes(self) -> int:
        b = self.f.elements * ELEM_BYTES[self.f.dtype]
        if self.bcast is not None:
            b += self.bcast.numel() * self.bcast.element_size()
        return int(b)

    @property
    def d2h_bytes(self) -> int:
        return int(self.out.numel() * self.out.element_size())

    def output_numpy(self) -> np.ndarray:
        return self.out.cpu().numpy().view(_NP_OUT[self.f.out_dtype])


class ConcurrentFusions:
    """Independent fusions (no buffer shared between them) each enqueued on a stream of its own, forked
    from the caller's stream by one event and joined back into it by one event per fusion: work queued
    on the caller's stream before run() happens before every fusion, and work queued after it sees all
    their outputs. A short fusion then fills the ramp and tail of a long one instead of waiting for it
    to drain, and the launches themselves overlap."""

    def __init__(self, fusions, device="cuda"):
        self.fusions = list(fusions)
        self.streams = [torch.cuda.Stream(device=device) for _ in self.fusions]
        self.fork = torch.cuda.Event()
        self.joins = [torch.cuda.Event() for _ in self.fusions]

    def run(self, stream=None):
        stream = torch.cuda.current_stream() if stream is None else stream
        self.fork.record(stream)
        for d, s, j in zip(self.fusions, self.streams, self.joins):
            s.wait_event(self.fork)
            d.run(stream=s)
            j.record(s)
        for j in self.joins:
            stream.wait_event(j)
