"""ctypes binding of libjolt (include/jolt.h): argument marshalling only.

Every function takes torch tensors (device memory, contiguous) or plain
integers, passes their addresses and the current CUDA stream to the C entry
point of the same name, and raises JoltError on a non-OK status.  No step of
the method runs here: all of it runs in libjolt's CUDA kernels.  The library
must have been built (python -m partial_tucker_rotated_st_b300.build); there
is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

FULL = -1
F32, BF16, F16 = 0, 1, 2
TOKEN_EXACT, TOKEN_RANDOMIZED = 0, 1
COST_FORMULA, COST_SERIALIZED = 0, 1
HEADER_BYTES = 256

STATUS = {0: "JOLT_OK", 1: "JOLT_ERR_INVALID", 2: "JOLT_ERR_INFEASIBLE", 3: "JOLT_ERR_NONFINITE",
          4: "JOLT_ERR_NOCONVERGE", 5: "JOLT_ERR_WORKSPACE", 6: "JOLT_ERR_CUDA",
          7: "JOLT_ERR_TOO_LARGE"}
(OK, ERR_INVALID, ERR_INFEASIBLE, ERR_NONFINITE, ERR_NOCONVERGE, ERR_WORKSPACE, ERR_CUDA,
 ERR_TOO_LARGE) = range(8)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libjolt.so")


class JoltError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)}")
        self.status = status


class JoltConfig(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("T", ctypes.c_int), ("D", ctypes.c_int),
                ("dtype", ctypes.c_int),
                ("n_rT", ctypes.c_int), ("rT", ctypes.c_int * 8),
                ("n_rd", ctypes.c_int), ("rd", ctypes.c_int * 8),
                ("n_b", ctypes.c_int), ("b", ctypes.c_int * 4),
                ("quant_block", ctypes.c_int), ("token_mode", ctypes.c_int),
                ("oversample", ctypes.c_int), ("power_iters", ctypes.c_int),
                ("cost_model", ctypes.c_int), ("align", ctypes.c_int)]


class JoltBlobDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("T", ctypes.c_int), ("D", ctypes.c_int),
                ("rT", ctypes.c_int), ("rd", ctypes.c_int), ("b", ctypes.c_int),
                ("block", ctypes.c_int), ("flags", ctypes.c_int),
                ("off_UT", ctypes.c_uint64), ("off_Ud", ctypes.c_uint64),
                ("off_G", ctypes.c_uint64), ("off_scale", ctypes.c_uint64),
                ("off_codes", ctypes.c_uint64), ("bytes", ctypes.c_uint64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


# C signatures: (name, restype, argtypes)
_P = ctypes.c_void_p
_SIG = {
    "jolt_num_candidates": (ctypes.c_int, [ctypes.POINTER(JoltConfig)]),
    "jolt_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(JoltConfig)]),
    "jolt_factor_group": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    "jolt_sweep_candidates": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P, _P, _P,
                                             ctypes.c_size_t, _P, _P, _P]),
    "jolt_allocate": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int64,
                                     ctypes.c_int, _P, _P, _P, _P]),
    "jolt_refine": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int64, _P, _P,
                                   _P]),
    "jolt_allocate_uniform": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_int64,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.c_int, _P,
                                             _P, _P]),
    "jolt_set_sweep_events": (ctypes.c_int, [_P, _P]),
    "jolt_set_factor_events": (ctypes.c_int, [ctypes.POINTER(_P)]),
    "jolt_set_solver_limits": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "jolt_model_candidates": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P,
                                             ctypes.c_size_t, ctypes.POINTER(ctypes.c_double),
                                             _P, _P]),
    "jolt_calibrate_eps2": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int32), ctypes.c_int, _P, _P,
                                           _P]),
    "jolt_blob_bytes": (ctypes.c_size_t, [ctypes.POINTER(JoltConfig), ctypes.c_int]),
    "jolt_encode": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P, _P, _P,
                                   ctypes.c_size_t, _P, _P, ctypes.c_size_t,
                                   ctypes.POINTER(JoltBlobDesc), _P]),
    "jolt_decode": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(JoltBlobDesc), _P,
                                   ctypes.c_size_t, _P, ctypes.c_int, _P]),
    "jolt_attend_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int]),
    "jolt_attend": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(JoltBlobDesc), _P,
                                   ctypes.c_size_t, _P, ctypes.c_int, ctypes.c_float, _P,
                                   ctypes.c_size_t, _P, _P]),
    "jolt_admit_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int]),
    "jolt_admit": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(JoltBlobDesc), _P, ctypes.c_size_t,
                                  _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
                                  ctypes.c_size_t, _P, ctypes.c_size_t,
                                  ctypes.POINTER(JoltBlobDesc), _P]),
    "jolt_sweep_candidates_noalloc": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P,
                                                     _P, _P, ctypes.c_size_t, _P, _P, _P]),
    "jolt_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "jolt_read_status": (ctypes.c_int, [ctypes.POINTER(JoltConfig), ctypes.c_int, _P, _P]),
    "jolt_decode_status": (ctypes.c_int, [_P]),
    "jolt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "jolt_launch_count": (ctypes.c_uint64, []),
}
EXPORTS = tuple(_SIG)

_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libjolt.so; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m partial_tucker_rotated_st_b300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def _check(fn: str, st: int):
    if st != OK:
        raise JoltError(fn, st)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def make_config(H: int, T: int, D: int, dtype: int, rT: Sequence[int], rd: Sequence[int],
                bits: Sequence[int], block: int, token_mode: int = TOKEN_EXACT,
                oversample: int = 8, power_iters: int = 2, cost_model: int = COST_FORMULA,
                align: int = 256) -> JoltConfig:
    c = JoltConfig()
    c.H, c.T, c.D, c.dtype = H, T, D, dtype
    c.n_rT = len(rT)
    for i, r in enumerate(rT):
        c.rT[i] = r
    c.n_rd = len(rd)
    for i, r in enumerate(rd):
        c.rd[i] = r
    c.n_b = len(bits)
    for i, b in enumerate(bits):
        c.b[i] = b
    c.quant_block = block
    c.token_mode = token_mode
    c.oversample = oversample
    c.power_iters = power_iters
    c.cost_model = cost_model
    c.align = align
    return c


def jolt_num_candidates(cfg: JoltConfig) -> int:
    return lib().jolt_num_candidates(ctypes.byref(cfg))


def jolt_workspace_size(cfg: JoltConfig) -> int:
    return lib().jolt_workspace_size(ctypes.byref(cfg))


def jolt_factor_group(cfg, n_units, X, sketch, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("jolt_factor_group", lib().jolt_factor_group(
        ctypes.byref(cfg), n_units, _ptr(X), _ptr(sketch), _ptr(ws), ws_bytes, _stream(stream)))


def jolt_sweep_candidates(cfg, n_units, X, signs, ws, dist, cost, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("jolt_sweep_candidates", lib().jolt_sweep_candidates(
        ctypes.byref(cfg), n_units, _ptr(X), _ptr(signs), _ptr(ws), ws_bytes, _ptr(dist),
        _ptr(cost), _stream(stream)))


def jolt_sweep_candidates_noalloc(cfg, n_units, X, signs, ws, dist, cost, ws_bytes=None,
                                  stream=None):
    """The sweep without any device allocation: its scratch is the library's
    static array (see include/jolt.h)."""
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("jolt_sweep_candidates_noalloc", lib().jolt_sweep_candidates_noalloc(
        ctypes.byref(cfg), n_units, _ptr(X), _ptr(signs), _ptr(ws), ws_bytes, _ptr(dist),
        _ptr(cost), _stream(stream)))


def jolt_noalloc_scratch_bytes() -> int:
    return lib().jolt_noalloc_scratch_bytes()


def jolt_allocate(n_units, n_cand, dist, cost, budget, align, choice, lam, status, stream=None):
    _check("jolt_allocate", lib().jolt_allocate(
        n_units, n_cand, _ptr(dist), _ptr(cost), int(budget), int(align), _ptr(choice),
        _ptr(lam), _ptr(status), _stream(stream)))


def jolt_refine(n_units, n_cand, dist, cost, budget, choice, n_swaps=None, stream=None):
    _check("jolt_refine", lib().jolt_refine(
        n_units, n_cand, _ptr(dist), _ptr(cost), int(budget), _ptr(choice), _ptr(n_swaps),
        _stream(stream)))


def jolt_allocate_uniform(n_units, n_cand, dist, cost, budget, cand_host: Sequence[int], choice,
                          status, stream=None):
    arr = (ctypes.c_int32 * len(cand_host))(*[int(c) for c in cand_host])
    _check("jolt_allocate_uniform", lib().jolt_allocate_uniform(
        n_units, n_cand, _ptr(dist), _ptr(cost), int(budget), arr, len(cand_host), _ptr(choice),
        _ptr(status), _stream(stream)))


def fixed_bit_candidates(cfg: JoltConfig, ib: int):
    """Flat indices of every rank pair at bit index ib of the config's grid."""
    return [(iT * cfg.n_rd + i_d) * cfg.n_b + ib for iT in range(cfg.n_rT) for i_d in range(cfg.n_rd)]


def fixed_rank_candidates(cfg: JoltConfig, iT: int, i_d: int):
    """Flat indices of every bit width at rank pair (iT, id) of the config's grid."""
    return [(iT * cfg.n_rd + i_d) * cfg.n_b + ib for ib in range(cfg.n_b)]


def jolt_set_sweep_events(start=None, stop=None):
    """Record two torch.cuda.Event (timing enabled, already created, i.e.
    recorded once) around the fused sweep kernel of later sweep calls; no
    arguments turns it off."""
    a = None if start is None else start.cuda_event
    b = None if stop is None else stop.cuda_event
    if (start is not None and not a) or (stop is not None and not b):
        raise ValueError("record the events once before passing them")
    _check("jolt_set_sweep_events", lib().jolt_set_sweep_events(a, b))


def jolt_set_factor_events(events=None):
    """Record five torch.cuda.Event (timing enabled, already recorded once) at
    the factor step's stage boundaries of later jolt_factor_group calls (see
    include/jolt.h); no argument turns it off."""
    if events is None:
        _check("jolt_set_factor_events", lib().jolt_set_factor_events(None))
        return
    if len(events) != 5 or any(not e.cuda_event for e in events):
        raise ValueError("five events, each recorded once before")
    arr = (_P * 5)(*[e.cuda_event for e in events])
    _check("jolt_set_factor_events", lib().jolt_set_factor_events(arr))


def jolt_model_candidates(cfg, n_units, ws, eps2_host: Sequence[float], dist, ws_bytes=None,
                          stream=None):
    """Modeled-error distortion table from the factor step's spectra."""
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    arr = (ctypes.c_double * max(1, len(eps2_host)))(*[float(e) for e in eps2_host])
    _check("jolt_model_candidates", lib().jolt_model_candidates(
        ctypes.byref(cfg), n_units, _ptr(ws), ws_bytes, arr, _ptr(dist), _stream(stream)))


def jolt_calibrate_eps2(rows, bits: Sequence[int], scratch, eps2, stream=None):
    """eps^2(b) of the codec's quantizer on Gaussian rows (n x D fp32, device)."""
    arr = (ctypes.c_int32 * len(bits))(*[int(b) for b in bits])
    _check("jolt_calibrate_eps2", lib().jolt_calibrate_eps2(
        _ptr(rows), rows.shape[0], rows.shape[1], arr, len(bits), _ptr(scratch), _ptr(eps2),
        _stream(stream)))


def jolt_blob_bytes(cfg: JoltConfig, cand: int) -> int:
    return lib().jolt_blob_bytes(ctypes.byref(cfg), cand)


def jolt_encode(cfg, n_units, X, signs, ws, choice_host: Sequence[int], blob, blob_stride,
                ws_bytes=None, stream=None):
    """Returns the list of JoltBlobDesc (host) of the serialized units."""
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    ch = (ctypes.c_int32 * n_units)(*[int(c) for c in choice_host])
    desc = (JoltBlobDesc * n_units)()
    _check("jolt_encode", lib().jolt_encode(
        ctypes.byref(cfg), n_units, _ptr(X), _ptr(signs), _ptr(ws), ws_bytes, ch, _ptr(blob),
        blob_stride, desc, _stream(stream)))
    return list(desc)


def jolt_decode(desc: Sequence[JoltBlobDesc], blob, blob_stride, xhat, out_dtype, stream=None):
    n = len(desc)
    arr = (JoltBlobDesc * n)(*desc)
    _check("jolt_decode", lib().jolt_decode(n, arr, _ptr(blob), blob_stride, _ptr(xhat),
                                            out_dtype, _stream(stream)))


def jolt_set_solver_limits(max_sweeps: int = 0, max_subspace_blocks: int = 0):
    """Iteration caps of the eigensolvers (0 restores a default)."""
    _check("jolt_set_solver_limits", lib().jolt_set_solver_limits(int(max_sweeps),
                                                                  int(max_subspace_blocks)))


def jolt_decode_status(stream=None) -> int:
    """Synchronises and returns the decoder's device status code (not
    raised): ERR_CUDA when a bounded wait of a decode gave up."""
    return lib().jolt_decode_status(_stream(stream))


def jolt_attend_workspace_size(n_groups, H, T, D, nq) -> int:
    return int(lib().jolt_attend_workspace_size(n_groups, H, T, D, nq))


def jolt_attend(desc: Sequence[JoltBlobDesc], blob, blob_stride, q, nq, scale, ws, out,
                ws_bytes=None, stream=None):
    """Attention over the compressed K (even slots) and V (odd slots) of each
    group; q and out are [groups][H][nq][D] fp32 device tensors."""
    n = len(desc)
    if n % 2:
        raise ValueError("desc holds K, V pairs")
    arr = (JoltBlobDesc * n)(*desc)
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("jolt_attend", lib().jolt_attend(n // 2, arr, _ptr(blob), blob_stride, _ptr(q), nq,
                                            float(scale), _ptr(ws), ws_bytes, _ptr(out),
                                            _stream(stream)))


def jolt_admit_workspace_size(n_units, H, tau, D) -> int:
    return int(lib().jolt_admit_workspace_size(n_units, H, tau, D))


def jolt_admit(desc_in: Sequence[JoltBlobDesc], blob_in, stride_in, X_new, x_dtype, tau, align,
               ws, blob_out, stride_out, ws_bytes=None, stream=None):
    """Admit tau new tokens (X_new [units][H][tau][D]) into each unit; returns
    the new blobs' descriptions."""
    n = len(desc_in)
    arr = (JoltBlobDesc * n)(*desc_in)
    out = (JoltBlobDesc * n)()
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("jolt_admit", lib().jolt_admit(n, arr, _ptr(blob_in), stride_in, _ptr(X_new), x_dtype,
                                          tau, align, _ptr(ws), ws_bytes, _ptr(blob_out),
                                          stride_out, out, _stream(stream)))
    return list(out)


def jolt_read_status(cfg, n_units, ws, stream=None) -> int:
    """Synchronises and returns the device status code (not raised)."""
    return lib().jolt_read_status(ctypes.byref(cfg), n_units, _ptr(ws), _stream(stream))


def jolt_status_string(s: int) -> str:
    return lib().jolt_status_string(s).decode()


def jolt_launch_count() -> int:
    return lib().jolt_launch_count()
