"""Shared GPU-side driver for the parity tests: seeded inputs from kvgen, the
CUDA path through the C-ABI (via the ctypes binding), results on the host."""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

import kvgen
from partial_tucker_rotated_st_b300 import build as jbuild
from partial_tucker_rotated_st_b300 import codec
from partial_tucker_rotated_st_b300 import jolt as J


def ensure_built():
    jbuild.build()


def host_inputs(w, units: Sequence[int]):
    xs = [kvgen.make_unit(w, u) for u in units]
    signs = np.stack([kvgen.make_signs(w, u) for u in units])
    sk = None
    if w.token_mode == "randomized":
        sk = np.stack([kvgen.make_sketch(w, u) for u in units])
    return xs, signs, sk


def to_device(w, xs, signs, sk):
    arr = np.ascontiguousarray(np.stack(xs))
    if w.dtype == "bf16":
        X = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
    else:
        X = torch.from_numpy(arr)
    X = X.cuda()
    S = torch.from_numpy(np.ascontiguousarray(signs)).cuda()
    K = None if sk is None else torch.from_numpy(np.ascontiguousarray(sk)).cuda()
    return X, S, K


@dataclasses.dataclass
class GpuRun:
    w: object
    units: List[int]
    X64: List[np.ndarray]
    signs: np.ndarray
    sketch: Optional[np.ndarray]
    dist: np.ndarray        # [U, n_cand]
    cost: np.ndarray
    status: int
    choice: Optional[np.ndarray] = None
    lam: Optional[float] = None
    alloc_status: Optional[int] = None
    blobs: Optional[List[bytes]] = None
    desc: Optional[list] = None
    xhat32: Optional[np.ndarray] = None
    xhat16: Optional[np.ndarray] = None   # bf16 bit patterns
    dev: Optional[tuple] = None           # (encoder, X, signs, sketch) on the device, if kept


def run(w, units: Optional[Sequence[int]] = None, budget: Optional[int] = None,
        serialize: bool = True, decode: bool = True, choice_override=None,
        refine: bool = False, keep: bool = False) -> GpuRun:
    ensure_built()
    units = list(range(w.n_units)) if units is None else list(units)
    xs, signs, sk = host_inputs(w, units)
    X, S, K = to_device(w, xs, signs, sk)
    cfg = codec.config_for(w)
    enc = codec.Encoder(cfg, len(units))
    enc.factor(X, K)
    enc.sweep(X, S)
    st = enc.status()
    r = GpuRun(w, units, [kvgen.unit_values_f64(w, x) for x in xs], signs, sk,
               enc.dist.cpu().numpy(), enc.cost.cpu().numpy(), st)
    if keep:
        r.dev = (enc, X, S, K)
    if budget is None:
        budget = int(w.budget_bytes * len(units) // w.n_units)
    enc.allocate(budget, refine=refine)
    torch.cuda.synchronize()
    r.choice = enc.choice.cpu().numpy().astype(np.int64)
    r.lam = float(enc.lam.cpu().item())
    r.alloc_status = int(enc.astat.cpu().item())
    if not serialize:
        return r
    ch = r.choice if choice_override is None else np.asarray(choice_override)
    desc = enc.serialize(X, S, [int(c) for c in ch])
    torch.cuda.synchronize()
    r.desc = desc
    blob = enc.blob.cpu().numpy()
    r.blobs = [blob[u, :desc[u].bytes].tobytes() for u in range(len(units))]
    if decode:
        x32 = codec.decode(desc, enc.blob, enc.stride, J.F32)
        x16 = codec.decode(desc, enc.blob, enc.stride, J.BF16)
        torch.cuda.synchronize()
        r.xhat32 = x32.cpu().numpy().astype(np.float64)
        r.xhat16 = x16.view(torch.int16).cpu().numpy().view(np.uint16)
    return r
