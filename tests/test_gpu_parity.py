"""GPU parity of the CUDA path (through the C-ABI) against the float64 oracle
on the same seeded inputs.

Tolerances (fixed by the benchmark spec of the path):
  * distortion tables and reconstructions: relative error <= 1e-3 with an
    absolute floor of 1e-6;
  * byte costs, blob layout and the allocation (when the oracle allocator is
    fed the GPU's own tables): bit-exact;
  * quantized codes, recomputed by the oracle from the GPU's stored factors:
    at most 1e-4 of them off, only by +-1, and only at rounding ties of the
    oracle's own values (fp32 against f64 residuals);
  * decode of a blob: the oracle's decode of the same blob to 1e-5 relative
    (identical stored factors); bf16 output within bf16 rounding of it.
"""
import numpy as np
import pytest

import kvgen
from oracle import jolt as oj
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-6

# Reduced workloads with the full-size generator: several tiles and a ragged
# tail in T, the subspace-iteration path (T > 128) and the randomized path.
SMALL = {
    "tiny": kvgen.WORKLOADS["tiny"],
    "mistral_small": kvgen.custom_workload("mistral_t1024", n_groups=2, H=8, T=160),
    "flash_small": kvgen.custom_workload("flash_t4096", n_groups=2, H=16, T=320),
}

_RUNS = {}


def gpu_run(name):
    if name not in _RUNS:
        _RUNS[name] = gh.run(SMALL[name])
    return _RUNS[name]


_ORACLE = {}


def oracle_tables(name):
    if name not in _ORACLE:
        w = SMALL[name]
        r = gpu_run(name)
        dists, facs = [], []
        for i, u in enumerate(r.units):
            sk = None if r.sketch is None else r.sketch[i].astype(np.float64)
            fac = oj.factorize(r.X64[i], w.rT, w.rd, w.token_mode, sk, w.power_iters)
            facs.append(fac)
            dists.append(oj.dist_table(r.X64[i], fac, r.signs[i], w.bits))
        _ORACLE[name] = (np.stack(dists).reshape(len(r.units), -1), facs)
    return _ORACLE[name]


def close(a, b, rel=REL, ab=ABS):
    a, b = np.asarray(a, float), np.asarray(b, float)
    return np.abs(a - b) <= np.maximum(rel * np.abs(b), ab)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_status_ok(name):
    assert gpu_run(name).status == 0


@pytest.mark.parametrize("name", sorted(SMALL))
def test_cost_table_bit_exact(name):
    w, r = SMALL[name], gpu_run(name)
    fac = oracle_tables(name)[1][0]
    ref = oj.cost_table(w.H, w.T, w.D, fac.rT_list, fac.rd_list, w.bits, w.block).reshape(-1)
    for u in range(len(r.units)):
        assert np.array_equal(r.cost[u], ref)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_distortion_table_matches_oracle(name):
    r = gpu_run(name)
    ref = oracle_tables(name)[0]
    ok = close(r.dist, ref)
    bad = np.argwhere(~ok)
    assert ok.all(), [(int(u), int(c), r.dist[u, c], ref[u, c]) for u, c in bad[:10]]


@pytest.mark.parametrize("name", sorted(SMALL))
def test_allocation_bit_exact_on_gpu_tables(name):
    w, r = SMALL[name], gpu_run(name)
    budget = int(w.budget_bytes * len(r.units) // w.n_units)
    z, lam, st = oj.allocate(r.dist, r.cost, budget, 256)
    assert list(z) == list(r.choice)
    assert lam == r.lam
    assert (st == oj.ALLOC_OK) == (r.alloc_status == 0)
    assert sum(int(r.cost[u, z[u]]) for u in range(len(z))) <= budget


@pytest.mark.parametrize("name", sorted(SMALL))
def test_allocation_total_distortion_vs_oracle(name):
    w, r = SMALL[name], gpu_run(name)
    budget = int(w.budget_bytes * len(r.units) // w.n_units)
    ref, _ = oracle_tables(name)
    zo, _, _ = oj.allocate(ref, r.cost, budget, 256)
    d_gpu = sum(r.dist[u, r.choice[u]] for u in range(len(r.units)))
    d_ora = sum(ref[u, zo[u]] for u in range(len(r.units)))
    assert abs(d_gpu - d_ora) <= 1e-3 * abs(d_ora) + 1e-9


@pytest.mark.parametrize("U,nc,coarse", [(16, 100, False), (16, 100, True), (3, 7, False),
                                         (40, 33, True), (300, 100, False)])
def test_allocate_synthetic_tables_bit_exact(U, nc, coarse):
    """The bisection allocator on seeded synthetic tables against the oracle's
    on the same tables: choice, lambda and status bit for bit, for a budget
    that z(0) meets, binding budgets, and one below the cheapest allocation.
    Dyadic distortions on a coarse grid make equal keys frequent (the tie
    rules decide); the coarse tables also repeat costs and whole (cost,
    distortion) pairs, so that candidates dominated only through the index
    tie-break occur; the (300, 100) tables do not fit in shared memory and are
    read from global memory."""
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    rng = np.random.default_rng(7000 + U * 131 + nc + 17 * coarse)
    if coarse:
        cost = rng.integers(1, 12, size=(U, nc)).astype(np.int64) * 4096
        dist = rng.integers(0, 8, size=(U, nc)).astype(np.float64) / 8.0
    else:
        cost = rng.integers(1, 1 << 18, size=(U, nc)).astype(np.int64) * 256
        dist = rng.integers(0, 64, size=(U, nc)).astype(np.float64) / 64.0
    cmin = int(cost.min(axis=1).sum())
    z0, _, _ = oj.allocate(dist, cost, 1 << 62, 256)
    c0 = int(oj.total_cost(cost, z0))
    budgets = [c0 + 4096, cmin + (c0 - cmin) // 3, cmin + (c0 - cmin) // 50, cmin, cmin - 1]
    dd, cc = torch.from_numpy(dist).cuda(), torch.from_numpy(cost).cuda()
    ch = torch.zeros(U, dtype=torch.int32, device="cuda")
    lam = torch.zeros(1, dtype=torch.float64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for budget in budgets:
        J.jolt_allocate(U, nc, dd, cc, budget, 256, ch, lam, st)
        torch.cuda.synchronize()
        zref, lref, sref = oj.allocate(dist, cost, budget, 256)
        assert list(ch.cpu().numpy()) == list(zref), budget
        assert float(lam.item()) == lref, (budget, float(lam.item()), lref)
        assert int(st.item()) == (J.OK if sref == oj.ALLOC_OK else J.ERR_INFEASIBLE)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_blob_header_and_scored_distortion(name):
    """The GPU's blob has the layout of its candidate, and the distortion of
    what the GPU's own decoder rebuilds from it is the GPU's table entry for
    that candidate (the sweep scores what is stored)."""
    w, r = SMALL[name], gpu_run(name)
    for i in range(len(r.units)):
        hd = oj.parse_header(r.blobs[i])
        c = int(r.choice[i])
        lay = oj.blob_layout(w.H, w.T, w.D, hd["rT"], hd["rd"], hd["b"], w.block)
        assert hd["bytes"] == lay["bytes"] == len(r.blobs[i]) == r.desc[i].bytes
        for k in ("UT", "Ud", "G", "scale", "codes"):
            assert hd[k] == lay[k]
        assert np.array_equal(hd["signs"], r.signs[i])
        assert r.cost[i, c] >= hd["bytes"]
        x = r.X64[i]
        e = x - r.xhat32[i].astype(np.float64)
        d = float(np.sum(e * e) / max(np.sum(x * x), 1e-300))
        assert close(r.dist[i, c], d, 1e-4, 1e-7), (i, c, r.dist[i, c], d)


def oracle_codes_from_blob(blob):
    """Codes and scales the oracle's quantizer gives for the blob's own
    stored factors."""
    hd = oj.parse_header(blob)
    H, T, D, rT, rd, b = hd["H"], hd["T"], hd["D"], hd["rT"], hd["rd"], hd["b"]

    def arr(off, n, shape):
        return np.frombuffer(blob, np.float16, n, off).astype(np.float64).reshape(shape)

    UT = None if hd["flags"] & 1 else arr(hd["UT"], T * rT, (T, rT))
    Ud = None if hd["flags"] & 2 else arr(hd["Ud"], D * rd, (D, rd))
    G = arr(hd["G"], H * rT * rd, (H, rT, rd))
    return oj.reconstruct(UT, G, Ud), hd


def check_codes_against_oracle(X64, blob, D):
    """The blob's scales and codes against the oracle's quantizer applied to
    the blob's own stored factors.

    The GPU forms each rotated residual in fp32 from values of the size of X,
    so its y carries an absolute error of a few fp32 steps of the row's |x|;
    a decision may differ only where the oracle's value sits that close to a
    rounding boundary (window: 1e-6 of the row's max |x|):
      * a scale s = fp16(m / qmax) by one fp16 step, where m / qmax is within
        the window / qmax of the midpoint of the two fp16 values;
      * a code by one, where y is within the window of a tie (k + 1/2) s.
    Returns (differing codes, codes compared)."""
    Xt, hd = oracle_codes_from_blob(blob)
    b = hd["b"]
    Q = oj.rotation_matrix(hd["signs"])
    Y = (X64 - Xt).reshape(-1, D) @ Q.T
    win = 1e-6 * np.max(np.abs(X64.reshape(-1, D)), axis=1)
    q_ref, s_ref = oj.quantize_blocks(Y, b)
    n = Y.size
    s_gpu = np.frombuffer(blob, np.float16, n // D, hd["scale"]).astype(np.float64)
    q_gpu = oj.unpack_codes(blob[hd["codes"]:hd["codes"] + n * b // 8], n, b).reshape(-1, D)
    qmax = 2 ** (b - 1) - 1
    ratio = np.max(np.abs(Y), axis=1) / qmax
    srow = s_gpu != s_ref
    for r in np.flatnonzero(srow):
        lo, hi = sorted((s_gpu[r], s_ref[r]))
        assert np.nextafter(np.float16(lo), np.float16(np.inf)) == np.float16(hi), r
        assert abs(ratio[r] - 0.5 * (lo + hi)) <= win[r] / qmax, r
    keep = ~srow
    qd = np.abs(q_gpu[keep] - q_ref[keep])
    assert qd.max(initial=0) <= 1
    s_k = s_ref[keep][:, None]
    z = Y[keep] / np.where(s_k > 0, s_k, 1.0)
    tie_dist = np.abs(np.abs(z - np.floor(z)) - 0.5) * s_k
    assert np.all((tie_dist <= win[keep][:, None])[qd != 0])
    return int(np.count_nonzero(qd)), int(qd.size)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_codes_match_oracle_quantizer(name):
    """Encode every b of one rank pair per unit and compare the codes with the
    oracle's quantizer applied to the same stored factors."""
    w = SMALL[name]
    r0 = gpu_run(name)
    nb, nd = len(w.bits), len(w.rd)
    bad = tot = 0
    for iT in range(len(w.rT)):
        # one rank pair per token rank, cycling through feature ranks
        idd = iT % nd
        choice = [((iT * nd + idd) * nb + nb - 1 - (u % 2)) for u in range(len(r0.units))]
        r = gh.run(w, choice_override=choice, decode=False)
        for i in range(len(r.units)):
            if oj.parse_header(r.blobs[i])["b"] == 0:
                continue
            nbad, n = check_codes_against_oracle(r.X64[i], r.blobs[i], w.D)
            bad += nbad
            tot += n
    assert tot > 0 and bad <= max(1e-4 * tot, 8)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_matches_oracle_decode(name):
    """The oracle serializes candidates of its own factors (cycling through
    every branch of the rebuild); the GPU decodes those blobs."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w, r = SMALL[name], gpu_run(name)
    facs = oracle_tables(name)[1]
    U = len(r.units)
    for rnd in range(3):
        blobs = []
        for u in range(U):
            iT, id_, ib = _ATT_CANDS[(rnd * U + u) % len(_ATT_CANDS)]
            f = facs[u]
            blobs.append(oj.encode_unit(r.X64[u], f, r.signs[u], f.rT_list[iT], f.rd_list[id_],
                                        w.bits[ib], w.block))
        dev, stride = _upload(blobs)
        desc = [_desc_of(b) for b in blobs]
        x32 = codec.decode(desc, dev, stride, J.F32).cpu().numpy()
        x16 = codec.decode(desc, dev, stride, J.BF16).view(torch.int16).cpu().numpy()
        for i in range(U):
            ref = oj.decode_unit(blobs[i])
            err = np.linalg.norm(x32[i] - ref) / max(np.linalg.norm(ref), 1e-30)
            assert err <= 1e-5
            # bf16 output: within bf16 rounding of the oracle's value plus the
            # fp32 arithmetic error of the reconstruction (absolute, at 1e-5
            # of the RMS value)
            g16 = kvgen.bf16_to_f32(x16[i].view(np.uint16)).astype(np.float64)
            rms = np.linalg.norm(ref) / np.sqrt(ref.size)
            assert np.all(np.abs(g16 - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * rms)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_distortion_properties(name):
    """Facts that hold whatever the factors: more bits never hurt, full
    ranks without residual reproduce X to fp16 rounding, rank monotonicity of
    the truncation error."""
    w, r = SMALL[name], gpu_run(name)
    nT, nd, nb = len(w.rT), len(w.rd), len(w.bits)
    d = r.dist.reshape(-1, nT, nd, nb)
    assert np.all(np.isfinite(d)) and np.all(d >= 0)
    assert np.all(np.diff(d, axis=3) <= 1e-9)
    assert np.all(d[:, -1, -1, 0] <= 1e-6)
    assert np.all(np.diff(d[..., 0], axis=1) <= 1e-6)
    assert np.all(np.diff(d[..., 0], axis=2) <= 1e-6)


def test_zero_unit_and_nonfinite_input():
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w = SMALL["mistral_small"]
    cfg = codec.config_for(w)
    enc = codec.Encoder(cfg, 2)
    X = torch.zeros(2, w.H, w.T, w.D, dtype=torch.bfloat16, device="cuda")
    S = torch.ones(2, w.D, dtype=torch.int8, device="cuda")
    enc.factor(X)
    enc.sweep(X, S)
    assert enc.status() == J.OK
    assert torch.all(enc.dist == 0)
    X[1, 3, 7, 5] = float("nan")
    enc.factor(X)
    enc.sweep(X, S)
    assert enc.status() == J.ERR_NONFINITE


@pytest.mark.parametrize("name", ["tiny", "mistral_small"])
def test_eigensolver_cap_reports_noconverge(name):
    """Every Jacobi solve capped at one sweep and the subspace iteration at
    one block: the factor step finishes (the loops are bounded compute) and
    reports JOLT_ERR_NOCONVERGE through the unit status; with the default caps
    restored the same input factors cleanly."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w = SMALL[name]
    xs, signs, sk = gh.host_inputs(w, range(w.n_units))
    X, S, K = gh.to_device(w, xs, signs, sk)
    cfg = codec.config_for(w)
    enc = codec.Encoder(cfg, w.n_units)
    try:
        J.jolt_set_solver_limits(1, 1)
        enc.factor(X, K)
        torch.cuda.synchronize()
        assert enc.status() == J.ERR_NOCONVERGE
    finally:
        J.jolt_set_solver_limits(0, 0)
    enc.factor(X, K)
    assert enc.status() == J.OK


def test_decode_status_clear_after_clean_decode():
    """jolt_decode_status reports no gave-up wait after ordinary decodes on the
    tensor-core decoder (bf16, D = 128), and reading it clears it."""
    from partial_tucker_rotated_st_b300 import jolt as J
    r = gpu_run("mistral_small")
    assert r.xhat16 is not None
    assert J.jolt_decode_status() == J.OK
    assert J.jolt_decode_status() == J.OK


def test_rank_deficient_feature_gram_matches_oracle():
    """A feature that is identically zero makes S_d singular: the Cholesky of
    the one-sided eigensolver meets a zero pivot, and that unit is solved by
    the two-sided Jacobi instead.  Its tables still match the oracle, and the
    unit next to it (definite S_d) is unaffected."""
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w = SMALL["mistral_small"]
    xs, signs, sk = gh.host_inputs(w, [0, 1])
    xs[0] = xs[0].copy()
    xs[0][:, :, 5] = 0
    X, S, K = gh.to_device(w, xs, signs, sk)
    enc = codec.Encoder(codec.config_for(w), 2)
    enc.factor(X, K)
    enc.sweep(X, S)
    assert enc.status() == J.OK
    dist = enc.dist.cpu().numpy()
    for i in range(2):
        x64 = kvgen.unit_values_f64(w, xs[i])
        fac = oj.factorize(x64, w.rT, w.rd, w.token_mode, None, w.power_iters)
        ref = oj.dist_table(x64, fac, signs[i], w.bits).reshape(-1)
        assert np.all(close(dist[i], ref)), i


@pytest.mark.parametrize("name", sorted(SMALL))
def test_refine_and_uniform_allocators_bit_exact_on_gpu_tables(name):
    """The greedy swap refinement and the uniform fixed-bit / fixed-rank
    allocators on the GPU, against the oracle's own on the same (GPU) tables:
    bit-exact choices and status."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w, r = SMALL[name], gpu_run(name)
    U = len(r.units)
    nc = r.dist.shape[1]
    dist = torch.from_numpy(r.dist).cuda()
    cost = torch.from_numpy(r.cost).cuda()
    budget = int(w.budget_bytes * U // w.n_units)
    # refinement after the bisection, from the GPU's own bisection result
    z0, _, st0 = oj.allocate(r.dist, r.cost, budget)
    ch = torch.from_numpy(np.asarray(r.choice, dtype=np.int32)).cuda()
    assert list(r.choice) == list(z0)
    ns = torch.zeros(1, dtype=torch.int32, device="cuda")
    J.jolt_refine(U, nc, dist, cost, budget, ch, ns)
    torch.cuda.synchronize()
    zref, nref = oj.refine_greedy(r.dist, r.cost, budget, z0)
    assert list(ch.cpu().numpy()) == list(zref) and int(ns.item()) == nref
    # a looser budget so that swaps actually happen
    zl, _, _ = oj.allocate(r.dist, r.cost, budget)
    loose = int(oj.total_cost(r.cost, zl)) + 3 * int(r.cost.max())
    ch = torch.from_numpy(np.asarray(zl, dtype=np.int32)).cuda()
    J.jolt_refine(U, nc, dist, cost, loose, ch, ns)
    torch.cuda.synchronize()
    zref, nref = oj.refine_greedy(r.dist, r.cost, loose, zl)
    assert list(ch.cpu().numpy()) == list(zref) and int(ns.item()) == nref
    # uniform baselines: fixed bits (every b of the grid) and fixed ranks
    cfg = codec.config_for(w)
    out = torch.zeros(U, dtype=torch.int32, device="cuda")
    stt = torch.zeros(1, dtype=torch.int32, device="cuda")
    lists = [J.fixed_bit_candidates(cfg, ib) for ib in range(cfg.n_b)]
    lists += [J.fixed_rank_candidates(cfg, iT, i_d) for iT in range(cfg.n_rT)
              for i_d in range(cfg.n_rd)]
    for cand in lists:
        for bud in (budget, budget // 4):
            J.jolt_allocate_uniform(U, nc, dist, cost, bud, cand, out, stt)
            torch.cuda.synchronize()
            zref, sref = oj.allocate_uniform(r.dist, r.cost, bud, cand)
            assert list(out.cpu().numpy()) == list(zref)
            assert int(stt.item()) == (J.OK if sref == oj.ALLOC_OK else J.ERR_INFEASIBLE)


def test_eps2_calibration_matches_oracle():
    """eps^2(b) of the codec's quantizer on the same seeded Gaussian rows."""
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    rng = np.random.default_rng(20260101)
    bits = [0, 2, 4, 8]
    for D in (32, 128):
        rows = rng.standard_normal((3000, D)).astype(np.float32)
        ref = oj.eps2_calibrate(rows.astype(np.float64), bits)
        scratch = torch.zeros(8, dtype=torch.float64, device="cuda")
        eps2 = torch.zeros(len(bits), dtype=torch.float64, device="cuda")
        J.jolt_calibrate_eps2(torch.from_numpy(rows).cuda(), bits, scratch, eps2)
        torch.cuda.synchronize()
        assert np.all(close(eps2.cpu().numpy(), ref, rel=1e-4, ab=0.0)), (D, eps2, ref)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_model_table_matches_oracle_and_allocates(name):
    """The modeled-error table from the GPU's spectra against the oracle's
    from its own (f64) factorization, at the path's tolerance; the bisection
    on the GPU's modeled table matches the oracle's bisection on it."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    w = SMALL[name]
    xs, signs, sk = gh.host_inputs(w, range(w.n_units))
    X, S, K = gh.to_device(w, xs, signs, sk)
    cfg = codec.config_for(w)
    U = w.n_units
    enc = codec.Encoder(cfg, U)
    enc.factor(X, K)
    eps2 = [1.0, 0.59, 0.0138, 4.2e-5][: len(w.bits)] if list(w.bits) == [0, 2, 4, 8] else \
        [1.0 if b == 0 else 4.0 ** (-b) for b in w.bits]
    md = torch.zeros(U, enc.ncand, dtype=torch.float64, device="cuda")
    J.jolt_model_candidates(cfg, U, enc.ws, eps2, md)
    assert enc.status() == J.OK
    md = md.cpu().numpy()
    for i in range(U):
        x64 = kvgen.unit_values_f64(w, xs[i])
        s_ = None if sk is None else sk[i].astype(np.float64)
        fac = oj.factorize(x64, w.rT, w.rd, w.token_mode, s_, w.power_iters)
        ref = oj.model_dist_table(fac, float(np.sum(x64 * x64)), w.bits, eps2)
        ok = close(md[i], ref)
        j = int(np.argmax(np.abs(md[i] - ref)))
        assert np.all(ok), (i, j, md[i][j], ref[j])
    enc.sweep(X, S)   # the cost table
    budget = int(w.budget_bytes * U // w.n_units)
    ch = torch.zeros(U, dtype=torch.int32, device="cuda")
    lam = torch.zeros(1, dtype=torch.float64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    J.jolt_allocate(U, enc.ncand, torch.from_numpy(md).cuda(), enc.cost, budget, cfg.align, ch,
                    lam, st)
    torch.cuda.synchronize()
    zref, lref, sref = oj.allocate(md, enc.cost.cpu().numpy(), budget, cfg.align)
    assert list(ch.cpu().numpy()) == list(zref) and float(lam.item()) == lref


# ------------------------------------------------ attention over the compressed cache
def _desc_of(blob):
    from partial_tucker_rotated_st_b300 import jolt as J
    hd = oj.parse_header(blob)
    d = J.JoltBlobDesc()
    d.H, d.T, d.D, d.rT, d.rd, d.b = hd["H"], hd["T"], hd["D"], hd["rT"], hd["rd"], hd["b"]
    d.block, d.flags = hd["block"], hd["flags"]
    d.off_UT, d.off_Ud, d.off_G = hd["UT"], hd["Ud"], hd["G"]
    d.off_scale, d.off_codes, d.bytes = hd["scale"], hd["codes"], hd["bytes"]
    return d


def _attend_gpu(blobs, q, scale):
    """jolt_attend on blobs uploaded from the host (K in even, V in odd slots)."""
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    stride = -(-max(len(b) for b in blobs) // 256) * 256
    host = np.zeros((len(blobs), stride), dtype=np.uint8)
    for i, b in enumerate(blobs):
        host[i, :len(b)] = np.frombuffer(b, dtype=np.uint8)
    dev = torch.from_numpy(host).cuda()
    G, H, nq, D = q.shape
    T = oj.parse_header(blobs[0])["T"]
    ws = torch.empty(J.jolt_attend_workspace_size(G, H, T, D, nq), dtype=torch.uint8, device="cuda")
    qd = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    out = torch.full((G, H, nq, D), float("nan"), dtype=torch.float32, device="cuda")
    J.jolt_attend([_desc_of(b) for b in blobs], dev, stride, qd, nq, scale, ws, out)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def _check_attention(blobs, q, scale):
    """Every output of the GPU against the oracle's attention over the two
    decoded blobs of each group.  fp32 bound: a score sums at most
    D + JOLT_ATTN_MAX_RANK products (the query-side coefficients as many
    again), so |ds| <= 4 (D + 128) 2^-24 (1 + scale |q| |K^_t|); the output
    moves by at most 2 max|ds| max|V^| through the softmax, plus the fp32
    sums over T tokens and D + 128 back-projection terms, (T + D + 128)
    2^-24 max|V^|.  Norm-wise the error must also stay below 1e-5."""
    out = _attend_gpu(blobs, q, scale)
    G, H, nq, D = q.shape
    q64 = q.astype(np.float64)
    for g in range(G):
        Kh, Vh = oj.decode_unit(blobs[2 * g]), oj.decode_unit(blobs[2 * g + 1])
        ref = oj.attention(q64[g], Kh, Vh, scale)
        T = Kh.shape[1]
        u = 2.0 ** -24
        E = scale * np.max(np.linalg.norm(q64[g], axis=2)) * np.max(np.linalg.norm(Kh, axis=2))
        vmax = np.max(np.abs(Vh))
        tol = (2 * 4 * (D + 128) * u * (1 + E) + (T + D + 128) * u) * vmax
        err = np.abs(out[g] - ref)
        assert np.all(np.isfinite(out[g]))
        j = np.unravel_index(np.argmax(err), err.shape)
        assert err[j] <= tol, (g, j, out[g][j], ref[j], tol)
        rel = np.linalg.norm(out[g] - ref) / max(np.linalg.norm(ref), 1e-30)
        assert rel <= 1e-5, (g, rel)


# candidate (iT, id, ib) of K and V per round: every branch of the fused
# rebuild (token rank truncated or whole, feature rank truncated or whole,
# every bit width, b = 0)
_ATT_CANDS = [(0, 0, 2), (-1, 0, 1), (1, -1, 3), (-1, -1, 0), (2, 1, 0), (0, -1, 2),
              (-1, 1, 2), (1, 1, 1), (-1, -1, 3), (3, 2, 2), (-1, 2, 3), (2, 0, 1)]


@pytest.mark.parametrize("name", sorted(SMALL))
def test_attend_matches_oracle_on_oracle_blobs(name):
    """The oracle serializes candidates of its own factors; the GPU attends
    over those blobs; the oracle attends over their decodes."""
    w, r = SMALL[name], gpu_run(name)
    facs = oracle_tables(name)[1]
    U = len(r.units)
    rng = np.random.default_rng(31)
    scale = 1.0 / np.sqrt(w.D)
    for rnd, nq in enumerate((1, 3, 4, 8)):
        blobs = []
        for u in range(U):
            iT, id_, ib = _ATT_CANDS[(rnd * U + u) % len(_ATT_CANDS)]
            f = facs[u]
            blobs.append(oj.encode_unit(r.X64[u], f, r.signs[u], f.rT_list[iT], f.rd_list[id_],
                                        w.bits[ib], w.block))
        q = rng.standard_normal((U // 2, w.H, nq, w.D)).astype(np.float32)
        _check_attention(blobs, q, scale)


def test_attend_full_size_random_blobs():
    """mistral_t1024's shape and the bench's launch (8 groups of
    [32, 1024, 128], 4 queries per head) on random blobs of mixed
    candidates, every output against the oracle."""
    w = kvgen.WORKLOADS["mistral_t1024"]
    rng = np.random.default_rng(32)
    rT = [oj.resolve(x, w.T) for x in w.rT]
    rd = [oj.resolve(x, w.D) for x in w.rd]
    blobs = []
    for u in range(w.n_units):
        signs = kvgen.make_signs(w, u)
        blobs.append(oj.random_blob(rng, w.H, w.T, w.D, rT[rng.integers(len(rT))],
                                    rd[rng.integers(len(rd))], w.bits[u % len(w.bits)], signs))
    q = rng.standard_normal((w.n_groups, w.H, 4, w.D)).astype(np.float32)
    _check_attention(blobs, q, 1.0 / np.sqrt(w.D))


@pytest.mark.parametrize("T,D,nq,rT,rd,b", [(1, 64, 2, 1, 8, 4), (129, 32, 8, 5, 4, 2),
                                            (257, 128, 5, 64, 128, 8), (200, 64, 1, 200, 64, 0),
                                            (129, 128, 3, 5, 8, 4), (130, 128, 2, 130, 7, 2)])
def test_attend_edge_shapes(T, D, nq, rT, rd, b):
    """One token; a last chunk of one or two tokens; odd ranks (the
    tensor-core chunk's unpaired row loads at D = 128); whole modes."""
    rng = np.random.default_rng(T + D)
    H = 3
    signs = np.where(rng.random(D) < 0.5, -1, 1).astype(np.int8)
    blobs = [oj.random_blob(rng, H, T, D, rT, rd, b, signs),
             oj.random_blob(rng, H, T, D, rT if rT < T else T, max(1, rd // 2) if rd < D else D,
                            {0: 2, 2: 4, 4: 8, 8: 2}[b], signs[::-1].copy())]
    q = rng.standard_normal((1, H, nq, D)).astype(np.float32)
    _check_attention(blobs, q, 0.5 / np.sqrt(D))
    # all-zero queries: uniform weights, the mean of V^ over the tokens
    out = _attend_gpu(blobs, np.zeros_like(q), 1.0)
    mean = oj.decode_unit(blobs[1]).mean(axis=1)
    assert np.allclose(out[0], np.repeat(mean[:, None, :], nq, axis=1), rtol=1e-5, atol=1e-5)


# ------------------------------------------------ admission of a new token block
def _upload(blobs):
    import torch
    stride = -(-max(len(b) for b in blobs) // 256) * 256
    host = np.zeros((len(blobs), stride), dtype=np.uint8)
    for i, b in enumerate(blobs):
        host[i, :len(b)] = np.frombuffer(b, dtype=np.uint8)
    return torch.from_numpy(host).cuda(), stride


def _admit_gpu(blobs, Xn_stored, dtype):
    """jolt_admit on oracle blobs uploaded from the host; the new blobs back
    as bytes."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    dev, stride = _upload(blobs)
    arr = np.ascontiguousarray(np.stack(Xn_stored))
    if dtype == "bf16":
        X = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        X = torch.from_numpy(arr).cuda()
    out, sout, desc = codec.admit([_desc_of(b) for b in blobs], dev, stride, X)
    torch.cuda.synchronize()
    host = out.cpu().numpy()
    return [host[i, :desc[i].bytes].tobytes() for i in range(len(blobs))], desc


def _compare_admitted(gpu, ref):
    """Header and the old tokens' sections bit for bit; the new fp16 rows of
    U_T or G: the GPU rounds a double-float value, the oracle an f64 one, so
    they agree except where the value sits within ~2^-40 of an fp16 tie
    (allowed: one fp16 step, at most 1e-3 of the rows' entries); new scales
    by at most one fp16 step and codes by at most one, at most 1e-4 of them
    (or 8), as for encode.  Returns (rows differing, codes differing, codes)."""
    hg, hr = oj.parse_header(gpu), oj.parse_header(ref)
    assert len(gpu) == len(ref) and gpu[:256] == ref[:256]
    H, T, D, rT, rd, b = hr["H"], hr["T"], hr["D"], hr["rT"], hr["rd"], hr["b"]
    f16 = lambda blob, off, n: np.frombuffer(blob, np.float16, n, off)
    nrow = 0
    if not hr["flags"] & 1:
        a, r = f16(gpu, hr["UT"], T * rT), f16(ref, hr["UT"], T * rT)
        nrow += _ulp_diffs(a, r)
    else:
        a, r = f16(gpu, hr["G"], H * T * rd), f16(ref, hr["G"], H * T * rd)
        nrow += _ulp_diffs(a, r)
    for k in ("Ud",):
        if hr[k]:
            assert gpu[hr[k]:hr[k] + 2 * D * rd] == ref[hr[k]:hr[k] + 2 * D * rd]
    if not hr["flags"] & 1:
        assert gpu[hr["G"]:hr["G"] + 2 * H * rT * rd] == ref[hr["G"]:hr["G"] + 2 * H * rT * rd]
    nbad = ncode = 0
    if b > 0:
        n = H * T * D
        sg, sr = f16(gpu, hr["scale"], H * T), f16(ref, hr["scale"], H * T)
        assert _ulp_diffs(sg, sr) <= max(1e-4 * sg.size, 8)
        qg = oj.unpack_codes(gpu[hr["codes"]:hr["codes"] + n * b // 8], n, b)
        qr = oj.unpack_codes(ref[hr["codes"]:hr["codes"] + n * b // 8], n, b)
        d = np.abs(qg - qr)
        assert d.max(initial=0) <= 1
        nbad, ncode = int(np.count_nonzero(d)), n
    return nrow, nbad, ncode


def _ulp_diffs(a, r):
    """Entries of two fp16 arrays that differ; every difference one fp16 step."""
    ai, ri = a.view(np.int16).astype(np.int64), r.view(np.int16).astype(np.int64)
    diff = ai != ri
    if diff.any():
        step = np.abs(np.nextafter(r[diff], np.float16(np.inf)).astype(np.float64) -
                      r[diff].astype(np.float64))
        assert np.all(np.abs(a[diff].astype(np.float64) - r[diff].astype(np.float64)) <= step * 1.0001)
    return int(np.count_nonzero(diff))


# (rT index, rd index, b index) per unit, cycling: truncated and whole token
# ranks, truncated and whole feature ranks, every bit width
_ADM_CANDS = [(0, 0, 2), (-1, 0, 1), (1, -1, 3), (-1, -1, 0), (2, 1, 2), (-1, 1, 3), (0, -1, 1),
              (-1, -1, 2)]


@pytest.mark.parametrize("name", sorted(SMALL))
def test_admit_matches_oracle(name):
    """The oracle encodes each unit (its own factors, candidates cycling
    through every branch); the GPU and the oracle admit tau new tokens of
    the same distribution (the generator with the next seed) into those
    blobs."""
    import dataclasses
    w, r = SMALL[name], gpu_run(name)
    facs = oracle_tables(name)[1]
    tau = 40
    wn = dataclasses.replace(w, seed=w.seed + 1)
    nrow = nbad = ncode = 0
    for rnd in range(2):
        blobs, refs, Xn = [], [], []
        for u in range(len(r.units)):
            iT, id_, ib = _ADM_CANDS[(rnd * len(r.units) + u) % len(_ADM_CANDS)]
            f = facs[u]
            blob = oj.encode_unit(r.X64[u], f, r.signs[u], f.rT_list[iT], f.rd_list[id_],
                                  w.bits[ib], w.block)
            xs = np.ascontiguousarray(kvgen.make_unit(wn, u)[:, :tau])
            blobs.append(blob)
            refs.append(oj.admit_unit(blob, kvgen.unit_values_f64(w, xs)))
            Xn.append(xs)
        outs, desc = _admit_gpu(blobs, Xn, w.dtype)
        for g, ref, d in zip(outs, refs, desc):
            assert d.bytes == len(ref)
            a, c, n = _compare_admitted(g, ref)
            nrow, nbad, ncode = nrow + a, nbad + c, ncode + n
    assert nbad <= max(1e-4 * ncode, 8), (nbad, ncode)
    assert nrow <= 8, nrow


def test_admit_full_size_random_blobs():
    """mistral_t1024's units ([32, 1024, 128]) as random blobs of mixed
    candidates, 128 new tokens each, every admitted blob against the
    oracle's."""
    w = kvgen.WORKLOADS["mistral_t1024"]
    rng = np.random.default_rng(51)
    tau = 128
    rT = [oj.resolve(x, w.T) for x in w.rT]
    rd = [oj.resolve(x, w.D) for x in w.rd]
    blobs, refs, Xn = [], [], []
    for u in range(w.n_units):
        blob = oj.random_blob(rng, w.H, w.T, w.D, rT[u % len(rT)], rd[(u // 2) % len(rd)],
                              w.bits[(u // 5) % len(w.bits)], kvgen.make_signs(w, u))
        x = rng.standard_normal((w.H, tau, w.D)).astype(np.float32)
        xb = kvgen.round_to_bf16(x)
        x64 = kvgen.bf16_to_f32(xb).astype(np.float64)
        blobs.append(blob)
        refs.append(oj.admit_unit(blob, x64))
        Xn.append(xb)
    outs, desc = _admit_gpu(blobs, Xn, "bf16")
    nrow = nbad = ncode = 0
    for g, r in zip(outs, refs):
        a, c, n = _compare_admitted(g, r)
        nrow, nbad, ncode = nrow + a, nbad + c, ncode + n
    assert nbad <= max(1e-4 * ncode, 8), (nbad, ncode)
    assert nrow <= 1e-3 * w.n_units * tau * 64, nrow


@pytest.mark.parametrize("rT,rd,b", [(64, 48, 4), (48, 64, 8), (40, 128, 2), (200, 64, 4),
                                     (64, 40, 0), (33, 17, 2)])
def test_decode_wide_ranks_and_ragged_tiles(rT, rd, b):
    """Truncated ranks above 32 (the decoder's 64-wide operand variant), odd
    ranks, a ragged last tile (T = 200), fp32 and bf16 output, against the
    oracle's decode of the same random blobs."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    rng = np.random.default_rng(rT * 7 + rd + b)
    H, T, D = 3, 200, 128
    blobs = [oj.random_blob(rng, H, T, D, rT, rd, b,
                            np.where(rng.random(D) < 0.5, -1, 1).astype(np.int8))
             for _ in range(2)]
    dev, stride = _upload(blobs)
    desc = [_desc_of(x) for x in blobs]
    x32 = codec.decode(desc, dev, stride, J.F32).cpu().numpy()
    x16 = codec.decode(desc, dev, stride, J.BF16).view(torch.int16).cpu().numpy()
    for i in range(2):
        ref = oj.decode_unit(blobs[i])
        err = np.linalg.norm(x32[i] - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err <= 1e-5, err
        g16 = kvgen.bf16_to_f32(x16[i].view(np.uint16)).astype(np.float64)
        rms = np.linalg.norm(ref) / np.sqrt(ref.size)
        assert np.all(np.abs(g16 - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * rms)


@pytest.mark.parametrize("tau", [1, 3])
def test_admit_single_tokens_and_zero_block(tau):
    """The decode-time case, one (or a few) new tokens per unit, and a block
    of zeros (zero residual, zero scales), against the oracle."""
    w, r = SMALL["mistral_small"], gpu_run("mistral_small")
    facs = oracle_tables("mistral_small")[1]
    import dataclasses
    wn = dataclasses.replace(w, seed=w.seed + 2)
    for zero in (False, True):
        blobs, refs, Xn = [], [], []
        for u in range(len(r.units)):
            iT, id_, ib = _ADM_CANDS[(u + 3 * tau) % len(_ADM_CANDS)]
            f = facs[u]
            blob = oj.encode_unit(r.X64[u], f, r.signs[u], f.rT_list[iT], f.rd_list[id_],
                                  w.bits[ib], w.block)
            xs = np.ascontiguousarray(kvgen.make_unit(wn, u)[:, :tau])
            if zero:
                xs = np.zeros_like(xs)
            blobs.append(blob)
            refs.append(oj.admit_unit(blob, kvgen.unit_values_f64(w, xs)))
            Xn.append(xs)
        outs, desc = _admit_gpu(blobs, Xn, w.dtype)
        for g, ref, d in zip(outs, refs, desc):
            assert d.bytes == len(ref)
            nrow, nbad, _ = _compare_admitted(g, ref)
            assert nrow == 0 and nbad == 0
