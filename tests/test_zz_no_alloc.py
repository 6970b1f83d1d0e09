"""The no-allocation sweep entry point, checked through the C ABI against
the regular one.

Some callers cannot allocate device memory; for them the library offers
jolt_sweep_candidates_noalloc, which keeps its scratch in a static device
array instead of the caller's workspace.  This file runs last (pytest orders
files by name) so that a failure here leaves every other test already run.
It passes on its own in a fresh process and after the rest of the suite: the
first call on the device sets up the array's address, and two calls in a row
must both give the regular entry point's tables.
"""
import numpy as np
import pytest

import kvgen
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-6


@pytest.mark.parametrize("case", ["tensor_core", "simt_f32_d32"])
def test_noalloc_sweep_matches_regular_sweep_twice(case):
    """bf16 D = 128 takes the tensor-core sweep; the fp32 D = 32 workload the
    SIMT sweep kernel with its per-tile partials in the static array."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    gh.ensure_built()
    if case == "tensor_core":
        w = kvgen.custom_workload("mistral_t1024", n_groups=2, H=8, T=160)
    else:
        w = kvgen.WORKLOADS["tiny"]
    xs, signs, sk = gh.host_inputs(w, range(w.n_units))
    X, S, K = gh.to_device(w, xs, signs, sk)
    cfg = codec.config_for(w)
    enc = codec.Encoder(cfg, w.n_units)
    enc.factor(X, K)
    enc.sweep(X, S)
    torch.cuda.synchronize()
    ref_d = enc.dist.cpu().numpy().copy()
    ref_c = enc.cost.cpu().numpy().copy()
    assert enc.status() == J.OK
    for _ in range(2):
        dist = torch.full_like(enc.dist, float("nan"))
        cost = torch.full_like(enc.cost, -1)
        J.jolt_sweep_candidates_noalloc(cfg, w.n_units, X, S, enc.ws, dist, cost)
        torch.cuda.synchronize()
        d = dist.cpu().numpy()
        assert np.array_equal(cost.cpu().numpy(), ref_c)
        assert np.all(np.abs(d - ref_d) <= np.maximum(REL * np.abs(ref_d), ABS))
    assert enc.status() == J.OK


def test_noalloc_rejects_batches_beyond_its_scratch():
    import ctypes
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    gh.ensure_built()
    w = kvgen.WORKLOADS["llama_t1024"]
    cfg = codec.config_for(w)
    per_unit = (w.T // 64) * w.H * (J.jolt_num_candidates(cfg) + 1) * 4
    n = J.jolt_noalloc_scratch_bytes() // per_unit + 1
    ws_bytes = n * J.jolt_workspace_size(cfg)
    st = J.lib().jolt_sweep_candidates_noalloc(ctypes.byref(cfg), n, 1 << 20, 1 << 20, 1 << 20,
                                               ws_bytes, 1 << 20, 1 << 20, None)
    assert st == J.ERR_TOO_LARGE
