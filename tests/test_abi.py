"""Host-side checks of the C-ABI library, no GPU needed: the shared object
loads and exports every function include/jolt.h declares; the host logic
(grid validation, candidate count, blob layout, workspace sizing) agrees with
the oracle's byte accounting; invalid arguments are rejected before any CUDA
call."""
import ctypes
import os
import re

import numpy as np
import pytest

import kvgen
from oracle import jolt as oj
from partial_tucker_rotated_st_b300 import build as jbuild
from partial_tucker_rotated_st_b300 import codec
from partial_tucker_rotated_st_b300 import jolt as J

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    jbuild.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "jolt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(jolt_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) == 25
    lib = ctypes.CDLL(J.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(J.EXPORTS)


def test_struct_sizes_match_c_layout():
    assert ctypes.sizeof(J.JoltConfig) == 4 * (4 + 1 + 8 + 1 + 8 + 1 + 4 + 6)
    assert ctypes.sizeof(J.JoltBlobDesc) == 8 * 4 + 6 * 8


@pytest.mark.parametrize("name", sorted(kvgen.WORKLOADS))
def test_blob_bytes_match_oracle_layout(name):
    w = kvgen.WORKLOADS[name]
    cfg = codec.config_for(w)
    rT = [oj.resolve(r, w.T) for r in w.rT]
    rd = [oj.resolve(r, w.D) for r in w.rd]
    cands = oj.candidate_list(rT, rd, w.bits)
    assert J.jolt_num_candidates(cfg) == len(cands)
    for c, (i, j, k) in enumerate(cands):
        lay = oj.blob_layout(w.H, w.T, w.D, rT[i], rd[j], w.bits[k], w.block)
        assert J.jolt_blob_bytes(cfg, c) == lay["bytes"]
    assert J.jolt_workspace_size(cfg) % 256 == 0 and J.jolt_workspace_size(cfg) > 0


def _cfg(**kw):
    w = kvgen.custom_workload("mistral_t1024", **kw) if kw else kvgen.WORKLOADS["mistral_t1024"]
    return codec.config_for(w)


@pytest.mark.parametrize("bad", [
    dict(D=96), dict(D=256), dict(block=64), dict(bits=(0, 3)), dict(bits=(4, 2)),
    dict(rT=(8, 4, kvgen.FULL)), dict(rT=(4, kvgen.FULL, 8)), dict(rT=(4, 2048)),
    dict(rd=(4, 128)), dict(rd=(4, 96)), dict(rT=(4, 80)),
    dict(token_mode="randomized", oversample=40),
])
def test_invalid_configs_rejected(bad):
    cfg = _cfg(**bad)
    assert J.jolt_num_candidates(cfg) == 0
    assert J.jolt_workspace_size(cfg) == 0
    st = J.lib().jolt_factor_group(ctypes.byref(cfg), 1, 1 << 20, None, 1 << 20, 1 << 40, None)
    assert st == J.ERR_INVALID


def test_null_and_workspace_errors_before_launch():
    cfg = _cfg()
    L = J.lib()
    ws = J.jolt_workspace_size(cfg)
    assert L.jolt_factor_group(ctypes.byref(cfg), 1, None, None, 1 << 20, ws, None) == J.ERR_INVALID
    assert L.jolt_factor_group(ctypes.byref(cfg), 0, 1 << 20, None, 1 << 20, ws, None) == J.ERR_INVALID
    assert L.jolt_factor_group(ctypes.byref(cfg), 2, 1 << 20, None, 1 << 20, ws, None) == J.ERR_WORKSPACE
    assert L.jolt_factor_group(ctypes.byref(cfg), 1, 1 << 20, None, None, ws, None) == J.ERR_WORKSPACE
    # misaligned workspace
    assert L.jolt_factor_group(ctypes.byref(cfg), 1, 1 << 20, None, (1 << 20) + 8, ws, None) == J.ERR_WORKSPACE
    # randomized mode needs the sketch
    rc = _cfg(token_mode="randomized")
    assert L.jolt_factor_group(ctypes.byref(rc), 1, 1 << 20, None, 1 << 20, 1 << 40, None) == J.ERR_INVALID
    assert L.jolt_allocate(0, 10, 1, 1, 100, 256, 1, 1, 1, None) == J.ERR_INVALID
    assert L.jolt_allocate(4, 10, None, 1, 100, 256, 1, 1, 1, None) == J.ERR_INVALID


def test_decode_rejects_inconsistent_descriptors():
    d = J.JoltBlobDesc()
    d.H, d.T, d.D, d.rT, d.rd, d.b, d.block = 4, 64, 32, 4, 4, 4, 32
    lay = oj.blob_layout(4, 64, 32, 4, 4, 4, 32)
    d.off_UT, d.off_Ud, d.off_G = lay["UT"], lay["Ud"], lay["G"]
    d.off_scale, d.off_codes, d.bytes = lay["scale"], lay["codes"], lay["bytes"]
    arr = (J.JoltBlobDesc * 1)(d)
    L = J.lib()
    # stride smaller than the blob
    assert L.jolt_decode(1, arr, 1 << 20, 256, 1 << 21, J.F32, None) == J.ERR_INVALID
    # bad dtype, bad b, bad block
    assert L.jolt_decode(1, arr, 1 << 20, 1 << 16, 1 << 21, J.F16, None) == J.ERR_INVALID
    arr[0].b = 3
    assert L.jolt_decode(1, arr, 1 << 20, 1 << 16, 1 << 21, J.F32, None) == J.ERR_INVALID
    arr[0].b = 4
    arr[0].block = 16
    assert L.jolt_decode(1, arr, 1 << 20, 1 << 16, 1 << 21, J.F32, None) == J.ERR_INVALID


def test_status_strings():
    for s in range(8):
        assert J.jolt_status_string(s) and "unknown" not in J.jolt_status_string(s)


def _attn_desc(H=4, T=300, D=128, rT=8, rd=16, b=4):
    lay = oj.blob_layout(H, T, D, rT, rd, b, D)
    d = J.JoltBlobDesc()
    d.H, d.T, d.D, d.rT, d.rd, d.b, d.block = H, T, D, rT, rd, b, D
    d.flags = (1 if rT == T else 0) | (2 if rd == D else 0)
    d.off_UT, d.off_Ud, d.off_G = lay["UT"], lay["Ud"], lay["G"]
    d.off_scale, d.off_codes, d.bytes = lay["scale"], lay["codes"], lay["bytes"]
    return d


def test_attend_workspace_size():
    # per (group, head, chunk of 128 tokens): nq * (max, sum, z[D], cv[128])
    # floats, padded to 256 bytes; then per (group, head) the query
    # coefficients, (128 + D) x nq' floats with nq' = nq rounded up to 1, 2, 4, 8
    def want(G, H, T, D, nq):
        part = G * H * (-(-T // 128)) * nq * (2 + D + 128) * 4
        npad = 1 if nq <= 1 else 2 if nq <= 2 else 4 if nq <= 4 else 8
        return -(-part // 256) * 256 + G * H * (128 + D) * npad * 4
    for args in [(3, 4, 300, 128, 4), (1, 1, 128, 32, 1), (2, 5, 1000, 64, 3), (1, 2, 1, 32, 8)]:
        assert J.jolt_attend_workspace_size(*args) == want(*args), args
    assert J.jolt_attend_workspace_size(1, 1, 128, 32, 9) == 0
    assert J.jolt_attend_workspace_size(0, 1, 128, 32, 1) == 0


@pytest.mark.parametrize("case", ["nq0", "nq9", "odd_blob", "stride", "mismatch", "rank",
                                  "bits", "block", "codes_align", "ws", "null"])
def test_attend_rejects_bad_arguments_before_launch(case):
    good = [_attn_desc(), _attn_desc(rT=300, rd=32, b=2)]
    desc = list(good)
    dev = 1 << 40                       # never dereferenced: validation fails first
    blob, stride, nq = dev, 1 << 20, 4
    ws_bytes = J.jolt_attend_workspace_size(1, 4, 300, 128, 4)
    q = out = ws = dev
    want = J.ERR_INVALID
    if case == "nq0":
        nq = 0
    elif case == "nq9":
        nq = 9
    elif case == "odd_blob":
        blob = dev + 16
    elif case == "stride":
        stride = (1 << 20) + 16
    elif case == "mismatch":
        desc[1] = _attn_desc(T=256)
    elif case == "rank":
        desc[0] = _attn_desc(rT=80)
    elif case == "bits":
        desc[0] = _attn_desc(b=3)
    elif case == "block":
        desc[0].block = 64
    elif case == "codes_align":
        desc[0].off_codes += 8
    elif case == "ws":
        ws_bytes -= 4
        want = J.ERR_WORKSPACE
    elif case == "null":
        q = None
    arr = (J.JoltBlobDesc * 2)(*desc)
    st = J.lib().jolt_attend(1, arr, blob, stride, q, nq, 0.125, ws, ws_bytes, out, None)
    assert st == want


def test_admit_workspace_size():
    # per unit: 256 bytes (signs), Y as double-float (H tau D 8), M in f64
    # (64 x 64 x 8), chain rows as double-float (H 64 D 8), padded to 256
    def want(U, H, tau, D):
        return U * (-(-(256 + H * tau * D * 8 + 64 * 64 * 8 + H * 64 * D * 8) // 256) * 256)
    for args in [(2, 4, 10, 32), (16, 32, 128, 128), (1, 3, 1, 64)]:
        assert J.jolt_admit_workspace_size(*args) == want(*args)
    assert J.jolt_admit_workspace_size(1, 4, 0, 32) == 0
    assert J.jolt_admit_workspace_size(1, 4, 8, 48) == 0


@pytest.mark.parametrize("case", ["tau0", "dtype", "align", "overlap", "mismatch", "rank",
                                  "ws", "null", "odd_out"])
def test_admit_rejects_bad_arguments_before_launch(case):
    desc = [_attn_desc(T=300, rT=8, rd=16, b=4), _attn_desc(T=300, rT=300, rd=32, b=2)]
    dev = 1 << 40
    blob_in, sin, blob_out, sout = dev, 1 << 20, dev + (4 << 20), 2 << 20
    tau, align, dt = 16, 256, J.BF16
    ws_bytes = J.jolt_admit_workspace_size(2, 4, 16, 128)
    X = ws = dev + (64 << 20)
    want = J.ERR_INVALID
    if case == "tau0":
        tau = 0
    elif case == "dtype":
        dt = J.F16
    elif case == "align":
        align = 96
    elif case == "overlap":
        blob_out = dev + (1 << 20)
    elif case == "mismatch":
        desc[1] = _attn_desc(T=256)
    elif case == "rank":
        desc[0] = _attn_desc(T=300, rT=80)
    elif case == "ws":
        ws_bytes -= 256
        want = J.ERR_WORKSPACE
    elif case == "null":
        X = None
    elif case == "odd_out":
        blob_out += 128
    arr = (J.JoltBlobDesc * 2)(*desc)
    out = (J.JoltBlobDesc * 2)()
    st = J.lib().jolt_admit(2, arr, blob_in, sin, X, dt, tau, align, ws, ws_bytes, blob_out, sout,
                            out, None)
    assert st == want


MAX_CAND = 8 * 8 * 4   # JOLT_MAX_CAND of include/jolt.h


def _bad_call(case):
    """One call that the library must reject before any CUDA call, and the
    status it must return.  Device pointers are fake and never dereferenced."""
    cfg = _cfg()
    L = J.lib()
    dev = 1 << 40
    wsz = J.jolt_workspace_size(cfg)
    ncand = J.jolt_num_candidates(cfg)
    i32 = lambda *v: (ctypes.c_int32 * max(len(v), 1))(*v)
    f64 = lambda *v: (ctypes.c_double * len(v))(*v)
    sweep_args = dict(n=1, X=dev, signs=dev, ws=dev, wsb=wsz, dist=dev, cost=dev)

    def sweep(fn, **kw):
        a = dict(sweep_args, **kw)
        return fn(ctypes.byref(cfg), a["n"], a["X"], a["signs"], a["ws"], a["wsb"], a["dist"],
                  a["cost"], None)

    def encode(n=1, choice=(0,), blob=dev, stride=1 << 26, ws=dev, wsb=wsz):
        desc = (J.JoltBlobDesc * max(n, 1))()
        return L.jolt_encode(ctypes.byref(cfg), n, dev, dev, ws, wsb,
                             i32(*choice) if choice is not None else None, blob, stride, desc,
                             None)

    cases = {
        "sweep_units0": (lambda: sweep(L.jolt_sweep_candidates, n=0), J.ERR_INVALID),
        "sweep_signs": (lambda: sweep(L.jolt_sweep_candidates, signs=None), J.ERR_INVALID),
        "sweep_dist": (lambda: sweep(L.jolt_sweep_candidates, dist=None), J.ERR_INVALID),
        "sweep_ws_small": (lambda: sweep(L.jolt_sweep_candidates, wsb=wsz - 256), J.ERR_WORKSPACE),
        "sweep_ws_align": (lambda: sweep(L.jolt_sweep_candidates, ws=dev + 8), J.ERR_WORKSPACE),
        "noalloc_cost": (lambda: sweep(L.jolt_sweep_candidates_noalloc, cost=None), J.ERR_INVALID),
        "noalloc_ws_small": (lambda: sweep(L.jolt_sweep_candidates_noalloc, wsb=wsz - 256),
                             J.ERR_WORKSPACE),
        "noalloc_too_large": (lambda: sweep(L.jolt_sweep_candidates_noalloc, n=65535,
                                            wsb=65535 * wsz), J.ERR_TOO_LARGE),
        "encode_units0": (lambda: encode(n=0), J.ERR_INVALID),
        "encode_choice_null": (lambda: encode(choice=None), J.ERR_INVALID),
        "encode_blob_align": (lambda: encode(blob=dev + 16), J.ERR_INVALID),
        "encode_stride_align": (lambda: encode(stride=(1 << 26) + 16), J.ERR_INVALID),
        "encode_stride_small": (lambda: encode(stride=256), J.ERR_INVALID),
        "encode_choice_range": (lambda: encode(choice=(ncand,)), J.ERR_INVALID),
        "encode_choice_negative": (lambda: encode(choice=(-1,)), J.ERR_INVALID),
        "encode_ws_small": (lambda: encode(wsb=wsz - 256), J.ERR_WORKSPACE),
        "refine_ncand": (lambda: L.jolt_refine(4, MAX_CAND + 1, dev, dev, 1 << 20, dev, dev, None),
                         J.ERR_INVALID),
        "refine_dist": (lambda: L.jolt_refine(4, 10, None, dev, 1 << 20, dev, dev, None),
                        J.ERR_INVALID),
        "uniform_cand_range": (lambda: L.jolt_allocate_uniform(4, 10, dev, dev, 1 << 20, i32(3, 10),
                                                               2, dev, dev, None), J.ERR_INVALID),
        "uniform_empty_list": (lambda: L.jolt_allocate_uniform(4, 10, dev, dev, 1 << 20, i32(3), 0,
                                                               dev, dev, None), J.ERR_INVALID),
        "allocate_align": (lambda: L.jolt_allocate(4, 10, dev, dev, 1 << 20, 0, dev, dev, dev, None),
                           J.ERR_INVALID),
        "model_eps2_negative": (lambda: L.jolt_model_candidates(ctypes.byref(cfg), 1, dev, wsz,
                                                                f64(1.0, -0.5, 0.01, 1e-4), dev,
                                                                None), J.ERR_INVALID),
        "model_eps2_nan": (lambda: L.jolt_model_candidates(ctypes.byref(cfg), 1, dev, wsz,
                                                           f64(1.0, 0.5, float("nan"), 1e-4), dev,
                                                           None), J.ERR_INVALID),
        "model_ws_small": (lambda: L.jolt_model_candidates(ctypes.byref(cfg), 1, dev, wsz - 256,
                                                           f64(1.0, 0.5, 0.01, 1e-4), dev, None),
                           J.ERR_WORKSPACE),
        "eps2_D": (lambda: L.jolt_calibrate_eps2(dev, 64, 96, i32(2, 4), 2, dev, dev, None),
                   J.ERR_INVALID),
        "eps2_bits": (lambda: L.jolt_calibrate_eps2(dev, 64, 128, i32(2, 3), 2, dev, dev, None),
                      J.ERR_INVALID),
        "eps2_nb": (lambda: L.jolt_calibrate_eps2(dev, 64, 128, i32(0, 2, 4, 8, 8), 5, dev, dev,
                                                  None), J.ERR_INVALID),
        "events_half": (lambda: L.jolt_set_sweep_events(dev, None), J.ERR_INVALID),
        "status_units0": (lambda: L.jolt_read_status(ctypes.byref(cfg), 0, dev, None),
                          J.ERR_INVALID),
        "status_ws_null": (lambda: L.jolt_read_status(ctypes.byref(cfg), 1, None, None),
                           J.ERR_INVALID),
    }
    return cases[case]


_BAD_CASES = ["sweep_units0", "sweep_signs", "sweep_dist", "sweep_ws_small", "sweep_ws_align",
              "noalloc_cost", "noalloc_ws_small", "noalloc_too_large", "encode_units0",
              "encode_choice_null", "encode_blob_align", "encode_stride_align",
              "encode_stride_small", "encode_choice_range", "encode_choice_negative",
              "encode_ws_small", "refine_ncand", "refine_dist", "uniform_cand_range",
              "uniform_empty_list", "allocate_align", "model_eps2_negative", "model_eps2_nan",
              "model_ws_small", "eps2_D", "eps2_bits", "eps2_nb", "events_half",
              "status_units0", "status_ws_null"]


@pytest.mark.parametrize("case", _BAD_CASES)
def test_entry_points_reject_bad_arguments_before_launch(case):
    call, want = _bad_call(case)
    n0 = J.jolt_launch_count()
    assert call() == want
    assert J.jolt_launch_count() == n0


def test_solver_limits_setter_is_host_only():
    """The eigensolver caps are plain host state: set, rejected, restored."""
    from partial_tucker_rotated_st_b300 import jolt as J
    lib = J.lib()
    assert lib.jolt_set_solver_limits(1, 1) == J.OK
    assert lib.jolt_set_solver_limits(-1, 0) == J.ERR_INVALID
    assert lib.jolt_set_solver_limits(0, -3) == J.ERR_INVALID
    assert lib.jolt_set_solver_limits(0, 0) == J.OK
