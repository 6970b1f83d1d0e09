"""Buffer management around the C entry points: one encoder for a batch of
units of one shape.  Device memory comes from torch; every step of the method
runs in libjolt's kernels (see jolt.py for the bindings).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch

from . import jolt as J

_DT = {"f32": J.F32, "bf16": J.BF16}
_TORCH_DT = {J.F32: torch.float32, J.BF16: torch.bfloat16}


def config_for(w) -> J.JoltConfig:
    """jolt_config of a workload description with fields H, T, D, dtype
    ("f32"/"bf16"), rT, rd, bits, block, token_mode ("exact"/"randomized"),
    oversample, power_iters."""
    return J.make_config(w.H, w.T, w.D, _DT[w.dtype], list(w.rT), list(w.rd), list(w.bits),
                         w.block,
                         J.TOKEN_RANDOMIZED if w.token_mode == "randomized" else J.TOKEN_EXACT,
                         getattr(w, "oversample", 8), getattr(w, "power_iters", 2))


@dataclasses.dataclass
class EncodeResult:
    dist: torch.Tensor          # [U, n_cand] f64 (device)
    cost: torch.Tensor          # [U, n_cand] int64 (device)
    choice: List[int]           # host
    lam: float
    alloc_status: int
    blob: torch.Tensor          # [U, stride] uint8 (device)
    desc: List[J.JoltBlobDesc]


class Encoder:
    """Owns the workspace and tables for n_units units of config cfg."""

    def __init__(self, cfg: J.JoltConfig, n_units: int, device="cuda"):
        self.cfg = cfg
        self.U = n_units
        self.device = torch.device(device)
        self.ncand = J.jolt_num_candidates(cfg)
        if self.ncand == 0:
            raise J.JoltError("jolt_num_candidates", J.ERR_INVALID)
        self.ws_unit = J.jolt_workspace_size(cfg)
        self.ws = torch.empty(n_units * self.ws_unit, dtype=torch.uint8, device=self.device)
        self.dist = torch.empty(n_units, self.ncand, dtype=torch.float64, device=self.device)
        self.cost = torch.empty(n_units, self.ncand, dtype=torch.int64, device=self.device)
        self.choice = torch.empty(n_units, dtype=torch.int32, device=self.device)
        self.lam = torch.empty(1, dtype=torch.float64, device=self.device)
        self.astat = torch.empty(1, dtype=torch.int32, device=self.device)
        self.nswap = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.stride = max(J.jolt_blob_bytes(cfg, c) for c in range(self.ncand))
        self.stride = (self.stride + 255) // 256 * 256
        self.blob = torch.empty(n_units, self.stride, dtype=torch.uint8, device=self.device)
        self.choice_host = torch.empty(n_units, dtype=torch.int32, pin_memory=True)

    def factor(self, X, sketch=None, stream=None):
        J.jolt_factor_group(self.cfg, self.U, X, sketch, self.ws, stream=stream)

    def sweep(self, X, signs, stream=None):
        J.jolt_sweep_candidates(self.cfg, self.U, X, signs, self.ws, self.dist, self.cost,
                                stream=stream)

    def allocate(self, budget: int, stream=None, refine: bool = False):
        """Bisection on lambda; with `refine`, then the greedy swaps."""
        J.jolt_allocate(self.U, self.ncand, self.dist, self.cost, budget, self.cfg.align,
                        self.choice, self.lam, self.astat, stream=stream)
        if refine:
            J.jolt_refine(self.U, self.ncand, self.dist, self.cost, budget, self.choice,
                          self.nswap, stream=stream)

    def serialize(self, X, signs, choice: Sequence[int], stream=None):
        return J.jolt_encode(self.cfg, self.U, X, signs, self.ws, choice, self.blob, self.stride,
                             stream=stream)

    def encode(self, X, signs, budget: int, sketch=None, stream=None,
               refine: bool = True) -> EncodeResult:
        """factor -> sweep -> allocate (bisection, then the greedy swaps unless
        `refine` is False) -> serialize; one small device-to-host copy of the
        chosen candidates sits between allocate and serialize."""
        self.factor(X, sketch, stream)
        self.sweep(X, signs, stream)
        self.allocate(budget, stream, refine=refine)
        self.choice_host.copy_(self.choice, non_blocking=True)
        s = torch.cuda.current_stream() if stream is None else stream
        s.synchronize()
        choice = self.choice_host.tolist()
        desc = self.serialize(X, signs, choice, stream)
        return EncodeResult(self.dist, self.cost, choice, float("nan"), -1, self.blob, desc)

    def blobs_to_host(self, desc: Sequence[J.JoltBlobDesc], out: torch.Tensor, stream=None) -> int:
        """Copy the serialized bytes of every unit (desc[u].bytes of slot u,
        not the slot padding) back to back into the 1-D uint8 host tensor
        `out` (pinned for an asynchronous copy); returns the byte count."""
        off = 0
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for u, d in enumerate(desc):
                n = int(d.bytes)
                out[off:off + n].copy_(self.blob[u, :n], non_blocking=True)
                off += n
        return off

    def status(self) -> int:
        return J.jolt_read_status(self.cfg, self.U, self.ws)


def decode(desc: Sequence[J.JoltBlobDesc], blob: torch.Tensor, stride: int,
           out_dtype: int = J.BF16, out: Optional[torch.Tensor] = None, stream=None):
    d0 = desc[0]
    if out is None:
        out = torch.empty(len(desc), d0.H, d0.T, d0.D, dtype=_TORCH_DT[out_dtype],
                          device=blob.device)
    J.jolt_decode(desc, blob, stride, out, out_dtype, stream=stream)
    return out


def attend(desc: Sequence[J.JoltBlobDesc], blob: torch.Tensor, stride: int, q: torch.Tensor,
           scale: float, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
           stream=None):
    """Attention of q [groups][H][nq][D] (fp32) over the compressed K (even
    blob slots) and V (odd slots) of each group; returns out (fp32, same
    shape as q).  ws: scratch of jolt_attend_workspace_size bytes (allocated
    here when None)."""
    G, H, nq, D = q.shape
    if ws is None:
        ws = torch.empty(J.jolt_attend_workspace_size(G, H, desc[0].T, D, nq), dtype=torch.uint8,
                         device=q.device)
    if out is None:
        out = torch.empty_like(q)
    J.jolt_attend(desc, blob, stride, q, nq, scale, ws, out, stream=stream)
    return out


def admit_stride(stride_in: int, H: int, tau: int, D: int, align: int = 256) -> int:
    """A blob slot size that holds any unit of slot size stride_in after tau
    more tokens: the new U_T rows or core rows, scales and codes, plus a
    section's alignment padding each."""
    extra = H * tau * (2 * D + 2 + D) + 2 * 64 * tau + 6 * align
    return -(-(stride_in + extra) // 256) * 256


def admit(desc: Sequence[J.JoltBlobDesc], blob: torch.Tensor, stride: int, X_new: torch.Tensor,
          align: int = 256, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
          stream=None):
    """Admit the new tokens X_new [units][H][tau][D] (bf16 or fp32) into the
    encoded units; returns (blob_out, stride_out, desc_out)."""
    U, H, tau, D = X_new.shape
    dt = J.BF16 if X_new.dtype == torch.bfloat16 else J.F32
    sout = admit_stride(stride, H, tau, D, align)
    if out is None:
        out = torch.empty(U, sout, dtype=torch.uint8, device=blob.device)
    if ws is None:
        ws = torch.empty(J.jolt_admit_workspace_size(U, H, tau, D), dtype=torch.uint8,
                         device=blob.device)
    d = J.jolt_admit(desc, blob, stride, X_new, dt, tau, align, ws, out, sout, stream=stream)
    return out, sout, d


def blob_desc(header: bytes) -> J.JoltBlobDesc:
    """The description of a serialized unit read from its 256-byte header
    (little-endian: magic, version, H, T, D, r_T, r_d, b, block, flags, then
    the section offsets and the total size)."""
    import struct
    magic, ver, H, T, D, rT, rd, b, block, flags = struct.unpack_from("<IIiiiiiiiI", header, 0)
    if magic != 0x544C4F4A:
        raise ValueError("not a JoLT blob header")
    offs = struct.unpack_from("<QQQQQQ", header, 40)
    d = J.JoltBlobDesc()
    d.H, d.T, d.D, d.rT, d.rd, d.b, d.block, d.flags = H, T, D, rT, rd, b, block, flags
    d.off_UT, d.off_Ud, d.off_G, d.off_scale, d.off_codes, d.bytes = offs
    return d
