"""Pins of the float64 oracle against facts fixed outside the oracle itself:
closed forms, library routines, textbook invariants, hand-worked values and
brute force.  CPU only.

What pins which oracle function:
  jacobi_eigh            numpy.linalg.eigh on random symmetric matrices;
                         2x2 closed form; diagonal input; residual/orthogonality
  sylvester_hadamard     closed form H[i, j] = (-1)^popcount(i & j)
  rotation_matrix        Q^T Q = I and ||Q R|| = ||R||  [P4 Key formulas]
  quantize_blocks        hand-worked golden rows; brute-force nearest level;
                         MSE ratio per +2 bits near 16  [P1 Stage 1]
  feature/token modes,   truncation error = sum of discarded eigenvalues
  cores (factorize)      (single mode) and = ||X||^2 - ||G||^2 (two modes)
  dist_table             full ranks + b = 0 -> ~0; b = 0 monotone in r_T, r_d
  token_mode_randomized  many power steps -> exact subspace
  cholesky_qr2           numpy.linalg.qr up to column signs
  cost_formula           hand arithmetic; fp16 footprint 268.4 MB [P5 Efficiency]
  blob_layout/codec      decode(encode) reproduces the scored candidate
  allocate               hand cases; brute force over all tiny allocations
  attention              torch's scaled_dot_product_attention (CPU, float64);
                         equal keys -> mean of V; T = 1 -> V; a dominant key;
                         joint permutation of the tokens
  pack_blob/random_blob  parse_header/decode_unit read back the drawn sections
  attend_group           = attention on decode_unit of each blob; full ranks,
                         b = 0 -> attention on the fp16-rounded tensors
  cholesky_solve_drop    numpy.linalg.solve on SPD systems; hand case with
                         zero pivots
  fold_in                exact ST-HOSVD factors: a token's own U_T row
  admit_unit             old tokens decode unchanged; tokens in the span of
                         the stored factors give zero residual; two blocks
                         admitted one after the other = one concatenated block;
                         whole modes, b = 0: the new tokens decode to fp16(X);
                         the rotated error of every new row is within half a
                         quantization step
"""
import itertools
import os

import numpy as np
import pytest

import kvgen
from oracle import jolt, run
from oracle.jacobi import jacobi_eigh, round_robin_rounds

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- Jacobi
@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 33, 64])
def test_jacobi_matches_library_eigh(n):
    rng = np.random.default_rng(n)
    A = rng.standard_normal((n, n))
    S = A + A.T
    w, V, _ = jacobi_eigh(S)
    ref = np.linalg.eigh(S)[0][::-1]
    scale = max(1.0, np.abs(ref).max())
    assert np.max(np.abs(w - ref)) <= 1e-12 * scale
    assert np.max(np.abs(V.T @ V - np.eye(n))) <= 1e-12
    assert np.max(np.abs(S @ V - V * w[None, :])) <= 1e-12 * scale


def test_jacobi_2x2_closed_form():
    a, b, c = 3.0, 1.5, -2.0
    S = np.array([[a, b], [b, c]])
    w, V, _ = jacobi_eigh(S)
    mid, rad = (a + c) / 2, np.hypot((a - c) / 2, b)
    assert np.allclose(w, [mid + rad, mid - rad], rtol=0, atol=1e-14)


def test_jacobi_diagonal_and_psd_gram():
    d = np.array([1.0, 5.0, 3.0, 3.0])
    w, V, sweeps = jacobi_eigh(np.diag(d))
    assert sweeps == 0 and list(w) == [5.0, 3.0, 3.0, 1.0]
    # ties broken by original index: the two 3.0 eigenvectors are e_2, e_3
    assert np.array_equal(np.abs(V[:, 1]), [0, 0, 1, 0])
    rng = np.random.default_rng(5)
    Z = rng.standard_normal((200, 20))
    w, V, _ = jacobi_eigh(Z.T @ Z)
    s = np.linalg.svd(Z, compute_uv=False)
    assert np.allclose(w, s ** 2, rtol=1e-12)


def test_round_robin_covers_every_pair_once():
    for n in (2, 5, 8, 13):
        seen = []
        for p, q in round_robin_rounds(n):
            assert len(set(p) | set(q)) == 2 * len(p)  # disjoint in a round
            seen += [tuple(sorted((int(a), int(b)))) for a, b in zip(p, q)]
        assert sorted(seen) == sorted(itertools.combinations(range(n), 2))


# ---------------------------------------------------------------- rotation
@pytest.mark.parametrize("D", [1, 2, 8, 32, 128])
def test_hadamard_closed_form(D):
    Hm = jolt.sylvester_hadamard(D)
    i = np.arange(D)
    pop = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    assert np.array_equal(Hm, (-1.0) ** pop)


def test_rotation_orthogonal_and_norm_preserving():
    rng = np.random.default_rng(0)
    sig = np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)
    Q = jolt.rotation_matrix(sig)
    assert np.max(np.abs(Q.T @ Q - np.eye(128))) <= 1e-14
    R = rng.standard_normal((500, 128)) * np.linspace(0.1, 10, 128)
    assert abs(np.linalg.norm(R @ Q.T) / np.linalg.norm(R) - 1) <= 1e-13


def test_rotation_spreads_outlier():
    # a single outlier coordinate is spread to equal magnitude on all D
    # coordinates: the Hadamard outlier-spreading the pages describe
    sig = kvgen.make_signs(kvgen.WORKLOADS["mistral_t1024"], 0)
    Q = jolt.rotation_matrix(sig)
    e = np.zeros(128)
    e[17] = 8.0
    assert np.allclose(np.abs(Q @ e), 8.0 / np.sqrt(128), atol=1e-14)


# ---------------------------------------------------------------- quantizer
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "quantizer_worked_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, y, s, q, packed = [p.strip() for p in line.split("|")]
            rows.append((int(b), np.array(y.split(), float), float(s),
                         np.array(q.split(), int), bytes(int(v) for v in packed.split())))
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_quantizer_golden(row):
    b, y, s_ref, q_ref, packed_ref = row
    q, s = jolt.quantize_blocks(y[None, :], b)
    assert s[0] == s_ref
    assert np.array_equal(q[0], q_ref)
    assert jolt.pack_codes(q[0], b) == packed_ref
    assert np.array_equal(jolt.unpack_codes(packed_ref, y.size, b), q_ref)


@pytest.mark.parametrize("b", [2, 4, 8])
def test_quantizer_nearest_level_brute_force(b):
    rng = np.random.default_rng(b)
    Y = rng.standard_normal((300, 16)) * rng.lognormal(0, 2, (300, 1))
    Y[0] = 0.0
    q, s = jolt.quantize_blocks(Y, b)
    levels = np.arange(-(2 ** (b - 1)), 2 ** (b - 1))
    for i in range(Y.shape[0]):
        if s[i] == 0:
            assert not q[i].any()
            continue
        err = np.abs(Y[i][:, None] - s[i] * levels[None, :])
        best = err.min(axis=1)
        mine = np.abs(Y[i] - s[i] * q[i])
        assert np.all(mine <= best + 1e-15 * np.abs(Y[i]).max())
        assert np.all(np.abs(q[i]) <= 2 ** (b - 1) - 1)  # clip never binds


def test_quantizer_mse_ratio_per_two_bits():
    # [P1 Stage 1]: MSE falls by 16.25-25.65x per two added bits against a
    # high-rate prediction of 16x; the ratio shrinks toward 16 as b grows
    rng = np.random.default_rng(11)
    Y = rng.standard_normal((20000, 128))
    mse = {}
    for b in (2, 4, 6, 8):
        q, s = jolt.quantize_blocks(Y, b)
        mse[b] = np.mean((Y - q * s[:, None]) ** 2)
    r = [mse[2] / mse[4], mse[4] / mse[6], mse[6] / mse[8]]
    assert 12 <= r[1] <= 32 and 12 <= r[2] <= 32
    assert r[0] > r[1] > r[2]


# ---------------------------------------------------------------- Tucker
def _small_tensor(H=3, T=40, D=16, seed=3):
    w = kvgen.custom_workload("tiny", H=H, T=T, D=D, cp_rank=6, noise=0.05,
                              outliers=(2,), seed=seed)
    return kvgen.make_unit_f64(w, 0), kvgen.make_unit_f64(w, 1)


@pytest.mark.parametrize("rd", [2, 5, 16])
def test_feature_truncation_error_is_discarded_eigenvalues(rd):
    for X in _small_tensor():
        w, V = jolt.feature_mode(X)
        P = V[:, :rd] @ V[:, :rd].T
        err = np.sum((X - np.einsum("htd,de->hte", X, P)) ** 2)
        assert abs(err - w[rd:].sum()) <= 1e-10 * np.sum(X * X)


@pytest.mark.parametrize("rT,rd", [(3, 16), (7, 4), (20, 9), (40, 3)])
def test_two_mode_st_hosvd_error(rT, rd):
    for X in _small_tensor():
        H, T, D = X.shape
        fac = jolt.factorize(X, [rT, jolt.FULL], [rd, jolt.FULL])
        rdr = jolt.resolve(rd, D)
        if rT < T:
            UT, G = fac.UT[rdr][:, :rT], fac.G[rdr][:, :rT, :]
        else:
            UT, G = None, fac.Y[rdr]
        Ud = None if rdr == D else fac.Ud[rdr]
        Xt = jolt.reconstruct(UT, G, Ud)
        err = np.sum((X - Xt) ** 2)
        nx = np.sum(X * X)
        feat_tail = fac.feat_eigvals[rdr:].sum()
        if rT < T:
            S_T = jolt.token_unfolding(fac.Y[rdr]) @ jolt.token_unfolding(fac.Y[rdr]).T
            tok_tail = np.linalg.eigvalsh(S_T)[::-1][rT:].sum()
        else:
            tok_tail = 0.0
        assert abs(err - (feat_tail + tok_tail)) <= 1e-10 * nx
        assert abs(err - (nx - np.sum(G * G))) <= 1e-10 * nx


def test_dual_and_direct_token_modes_agree():
    X, _ = _small_tensor(H=2, T=30, D=8)
    Y = np.einsum("htd,dj->htj", X, jolt.feature_mode(X)[1][:, :4])  # K = 8 < T
    w1, U1 = jolt.token_mode_exact(Y, 6)
    A = jolt.token_unfolding(Y)
    w2, U2, _ = jacobi_eigh(A @ A.T)
    assert np.allclose(w1, w2[:6], rtol=1e-12)
    assert np.max(np.abs(U1 @ U1.T - U2[:, :6] @ U2[:, :6].T)) <= 1e-10


def _tiny_tables():
    w = kvgen.WORKLOADS["tiny"]
    Xs = [kvgen.unit_values_f64(w, kvgen.make_unit(w, u)) for u in range(w.n_units)]
    S = [kvgen.make_signs(w, u) for u in range(w.n_units)]
    return w, Xs, S, run.encode_units(Xs, S, w.rT, w.rd, w.bits, w.block, w.budget_bytes)


_TINY = {}


def tiny():
    if not _TINY:
        _TINY["v"] = _tiny_tables()
    return _TINY["v"]


def test_full_ranks_b0_reproduce_x():
    w, Xs, S, r = tiny()
    assert np.all(r.dist[:, -1, -1, 0] <= 1e-6)


def test_b0_distortion_monotone_in_ranks():
    w, Xs, S, r = tiny()
    d0 = r.dist[..., 0]
    assert np.all(np.diff(d0, axis=1) <= 1e-7)  # in r_T
    assert np.all(np.diff(d0, axis=2) <= 1e-7)  # in r_d


def test_residual_bits_lower_distortion():
    w, Xs, S, r = tiny()
    assert np.all(np.diff(r.dist, axis=3) < 0)


def test_randomized_converges_to_exact():
    w = kvgen.custom_workload("tiny", H=4, T=96, D=32, cp_rank=6, noise=0.001,
                              rT=(2, 4, jolt.FULL), rd=(4, 8, jolt.FULL))
    X = kvgen.make_unit_f64(w, 1)
    sk = kvgen.make_sketch(w, 1).astype(np.float64)
    ex = jolt.factorize(X, w.rT, w.rd, "exact")
    rz = jolt.factorize(X, w.rT, w.rd, "randomized", sk, power_iters=30)
    for rd in ex.rd_list:
        for k in (2, 4):
            Pe = ex.UT[rd][:, :k] @ ex.UT[rd][:, :k].T
            Pr = rz.UT[rd][:, :k] @ rz.UT[rd][:, :k].T
            assert np.max(np.abs(Pe - Pr)) <= 1e-8


def test_cholesky_qr2_matches_library_qr():
    rng = np.random.default_rng(2)
    Z = rng.standard_normal((300, 12)) @ np.diag(np.logspace(0, 3, 12))
    Q = jolt.cholesky_qr2(Z)
    Qn, Rn = np.linalg.qr(Z)
    Qn = Qn * np.sign(np.diag(Rn))[None, :]
    assert np.max(np.abs(Q - Qn)) <= 1e-10
    G = rng.standard_normal((9, 9))
    G = G @ G.T + np.eye(9)
    assert np.allclose(jolt.cholesky_lower(G), np.linalg.cholesky(G), atol=1e-13)


# ---------------------------------------------------------------- cost / codec
def test_cost_formula_hand_values():
    # tiny unit H=4, T=64, D=32, block 32:
    # (4,4,0): 2*4*(4*64 + 4*4 + 4*32) = 3200 -> 3328 aligned, + 256 header
    assert jolt.cost_formula(4, 64, 32, 4, 4, 0, 32) == 3584
    # (4,4,4): 3328 + 4*8192/8 = 4096 + 2*8192/32 = 512 + 256 = 8192
    assert jolt.cost_formula(4, 64, 32, 4, 4, 4, 32) == 8192
    # Mistral unit H=32, T=1024, D=128, (32,32,4):
    # 2*32*(32768 + 1024 + 4096) = 2424832; codes 2097152; scales 65536
    assert jolt.cost_formula(32, 1024, 128, 32, 32, 4, 128) == 2424832 + 2097152 + 65536 + 256


def test_fp16_footprint_matches_pages():
    # [P5 Efficiency]: Mistral KV at ctx 2048 is 268.4 MB in fp16
    w = kvgen.WORKLOADS["mistral_t2048"]
    assert w.fp16_bytes == 32 * 8 * 128 * 2048 * 2 * 2 == 268435456


def test_blob_never_exceeds_formula_cost():
    for w in kvgen.WORKLOADS.values():
        rT = [jolt.resolve(r, w.T) for r in w.rT]
        rd = [jolt.resolve(r, w.D) for r in w.rd]
        f = jolt.cost_table(w.H, w.T, w.D, rT, rd, w.bits, w.block, "formula")
        s = jolt.cost_table(w.H, w.T, w.D, rT, rd, w.bits, w.block, "serialized")
        assert np.all(s <= f)


def test_codec_round_trip_reproduces_scored_candidate():
    w, Xs, S, r = tiny()
    for u in range(w.n_units):
        xh = jolt.decode_unit(r.blobs[u])
        d = jolt.distortion(Xs[u], xh)
        assert d == pytest.approx(r.dist[u].reshape(-1)[r.choice[u]], rel=1e-12, abs=1e-15)
        hd = jolt.parse_header(r.blobs[u])
        assert np.array_equal(hd["signs"], S[u])
        assert hd["bytes"] == len(r.blobs[u]) <= r.cost[u].reshape(-1)[r.choice[u]]
    # every candidate of one unit round-trips
    X, fac = Xs[1], r.factors[1]
    for iT, idd, ib in jolt.candidate_list(fac.rT_list, fac.rd_list, w.bits):
        blob = jolt.encode_unit(X, fac, S[1], fac.rT_list[iT], fac.rd_list[idd], w.bits[ib], w.block)
        assert jolt.distortion(X, jolt.decode_unit(blob)) == pytest.approx(
            r.dist[1, iT, idd, ib], rel=1e-12, abs=1e-15)


def test_zero_unit():
    X = np.zeros((2, 16, 8))
    fac = jolt.factorize(X, [4, jolt.FULL], [2, jolt.FULL])
    d = jolt.dist_table(X, fac, np.ones(8, np.int8))
    assert np.all(d == 0.0)


# ---------------------------------------------------------------- allocation
def test_allocate_hand_case():
    dist = np.array([[1.0, 0.1], [0.5, 0.4]])
    cost = np.array([[100, 300], [100, 200]])
    # align = 1: stop only on an exact fit (the early stop within one
    # alignment block would accept the first feasible point here)
    z, lam, st = jolt.allocate(dist, cost, 400, align=1)
    assert st == jolt.ALLOC_OK and list(z) == [1, 0]
    assert 0.001 < lam < 0.0045
    z, lam, st = jolt.allocate(dist, cost, 10 ** 6)
    assert list(z) == [1, 1] and lam == 0.0
    z, lam, st = jolt.allocate(dist, cost, 150)
    assert st == jolt.ALLOC_INFEASIBLE and list(z) == [0, 0]


def test_allocate_brute_force_tiny():
    w, Xs, S, r = tiny()
    U = w.n_units
    dist = r.dist.reshape(U, -1)
    cost = r.cost.reshape(U, -1)
    z, lam, st = jolt.allocate(dist, cost, w.budget_bytes)
    assert st == jolt.ALLOC_OK
    Dz = sum(dist[u, z[u]] for u in range(U))
    Cz = sum(int(cost[u, z[u]]) for u in range(U))
    assert Cz <= w.budget_bytes
    # all 80^4 allocations, as (units 0,1) x (units 2,3)
    d01 = (dist[0][:, None] + dist[1][None, :]).reshape(-1)
    c01 = (cost[0][:, None] + cost[1][None, :]).reshape(-1)
    d23 = (dist[2][:, None] + dist[3][None, :]).reshape(-1)
    c23 = (cost[2][:, None] + cost[3][None, :]).reshape(-1)
    order = np.argsort(c23, kind="stable")
    c23s, d23min = c23[order], np.minimum.accumulate(d23[order])

    def best_at(limit):
        k = np.searchsorted(c23s, limit - c01, side="right") - 1
        ok = k >= 0
        return np.min(np.where(ok, d01 + d23min[np.maximum(k, 0)], np.inf))

    # on the lower convex hull: nothing at most as costly is better
    assert best_at(Cz) >= Dz - 1e-12
    # the duality gap to the true optimum at the budget is reported, not pinned
    gap = Dz - best_at(w.budget_bytes)
    assert gap >= -1e-12


def test_fix_signs_rule():
    V = np.array([[0.6, -0.8, 0.0], [-0.8, -0.6, 0.5], [0.0, 0.0, -0.5]])
    F = jolt.fix_signs(V)
    # column 0: |-0.8| largest -> flipped; column 1: |-0.8| -> flipped;
    # column 2: tie 0.5 / -0.5 -> the lower index (+0.5) decides, unchanged
    assert np.array_equal(F, np.array([[-0.6, 0.8, 0.0], [0.8, 0.6, 0.5], [0.0, 0.0, -0.5]]))
    w, V2 = jolt.feature_mode(_small_tensor()[0])
    assert np.all(V2[np.argmax(np.abs(V2), 0), np.arange(V2.shape[1])] > 0)


def test_refine_greedy_hand_case():
    # unit 0 can buy 0.5 of distortion for 100 bytes (rate 0.005), unit 1
    # 0.3 for 50 bytes (rate 0.006): with 120 bytes of slack only unit 1's
    # swap is taken first, and then unit 0's no longer fits
    dist = np.array([[1.0, 0.5], [0.9, 0.6]])
    cost = np.array([[100, 200], [100, 150]])
    z, n = jolt.refine_greedy(dist, cost, 320, np.array([0, 0]))
    assert list(z) == [0, 1] and n == 1
    # with 150 bytes of slack both swaps fit, the higher rate first
    z, n = jolt.refine_greedy(dist, cost, 350, np.array([0, 0]))
    assert list(z) == [1, 1] and n == 2
    # a swap that adds bytes but no distortion reduction is never taken
    dist2 = np.array([[0.5, 0.5]])
    cost2 = np.array([[100, 101]])
    z, n = jolt.refine_greedy(dist2, cost2, 10 ** 6, np.array([0]))
    assert list(z) == [0] and n == 0


def test_refine_greedy_properties():
    """Checked by enumeration: the result keeps the budget, never raises the
    total distortion, and at the end no single swap that adds bytes and
    lowers a unit's distortion still fits in the slack."""
    rng = np.random.default_rng(7)
    for trial in range(5):
        dist = rng.random((5, 12))
        cost = rng.integers(50, 400, (5, 12))
        z0 = np.argmin(cost, axis=1)
        budget = int(cost[np.arange(5), z0].sum()) + int(rng.integers(0, 900))
        z, n = jolt.refine_greedy(dist, cost, budget, z0)
        assert jolt.total_cost(cost, z) <= budget
        assert dist[np.arange(5), z].sum() <= dist[np.arange(5), z0].sum()
        slack = budget - jolt.total_cost(cost, z)
        for u in range(5):
            for c in range(12):
                dc = cost[u, c] - cost[u, z[u]]
                assert not (0 < dc <= slack and dist[u, c] < dist[u, z[u]])


def test_allocate_uniform_hand_case():
    # three candidates shared by two units: 1 is the best that fits
    dist = np.array([[0.1, 0.3, 0.9], [0.2, 0.2, 0.8]])
    cost = np.array([[500, 200, 50], [500, 250, 60]])
    z, st = jolt.allocate_uniform(dist, cost, 460, [0, 1, 2])
    assert st == jolt.ALLOC_OK and list(z) == [1, 1]
    z, st = jolt.allocate_uniform(dist, cost, 100, [0, 1, 2])
    assert st == jolt.ALLOC_INFEASIBLE and list(z) == [2, 2]
    assert jolt.fixed_bit_candidates(2, 3, 4, 2) == [2, 6, 10, 14, 18, 22]
    assert jolt.fixed_rank_candidates(2, 3, 4, 1, 2) == [20, 21, 22, 23]


# ---------------------------------------------------------------- modeled error
@pytest.mark.parametrize("rT,rd", [(3, 16), (7, 4), (20, 9), (40, 3), (40, 16)])
def test_tail_energy_is_the_unrounded_truncation_error(rT, rd):
    """tau from the spectra equals ||X - X~||^2 reconstructed from the
    unrounded factors (measured directly, not through the spectra)."""
    for X in _small_tensor():
        H, T, D = X.shape
        fac = jolt.factorize(X, [rT, jolt.FULL], [rd, jolt.FULL])
        rdr, rTr = jolt.resolve(rd, D), jolt.resolve(rT, T)
        if rTr < T:
            UT, G = fac.UT[rdr][:, :rTr], fac.G[rdr][:, :rTr, :]
        else:
            UT, G = None, fac.Y[rdr]
        Ud = None if rdr == D else fac.Ud[rdr]
        err = np.sum((X - jolt.reconstruct(UT, G, Ud)) ** 2)
        nx = float(np.sum(X * X))
        assert abs(jolt.tail_energy(fac, rTr, rdr, nx) - err) <= 1e-9 * nx


def test_eps2_uniform_noise_approximation():
    """For fine steps the rounding error of a row is uniform on [-s/2, s/2]:
    eps^2(b) ~ E[s^2] / 12 / E[y^2] with s = max|y| / (2^(b-1) - 1).  Checked at
    b = 8 against that closed form, within the fp16 rounding of s and the
    Monte Carlo spread; eps^2(0) = 1 and eps^2 falls with b."""
    rng = np.random.default_rng(11)
    rows = rng.standard_normal((4000, 128))
    e = jolt.eps2_calibrate(rows, [0, 2, 4, 8])
    assert e[0] == 1.0 and e[0] > e[1] > e[2] > e[3] > 0
    m2 = np.mean(np.max(np.abs(rows), axis=1) ** 2)
    approx = m2 / 127.0 ** 2 / 12.0 / np.mean(rows * rows)
    assert abs(e[3] / approx - 1.0) < 0.05


def test_model_dist_table_layout_and_scaling():
    X, _ = _small_tensor()
    H, T, D = X.shape
    fac = jolt.factorize(X, [4, jolt.FULL], [4, jolt.FULL])
    nx = float(np.sum(X * X))
    eps2 = np.array([1.0, 0.5, 0.01, 1e-4])
    t = jolt.model_dist_table(fac, nx, [0, 2, 4, 8], eps2).reshape(2, 2, 4)
    # (T, D) reproduces X exactly; b = 0 is the bare tail; b > 0 scales it
    assert np.all(t[1, 1] == 0.0)
    assert abs(t[0, 0, 0] - jolt.tail_energy(fac, 4, 4, nx) / nx) <= 1e-15
    assert np.allclose(t[0, 0, 1:], eps2[1:] * t[0, 0, 0], rtol=1e-15)
    assert abs(t[1, 0, 0] - fac.feat_eigvals[4:].sum() / nx) <= 1e-12
    assert np.all(jolt.model_dist_table(fac, 0.0, [0, 2, 4, 8], eps2) == 0.0)


# ---------------------------------------------------------------- attention
def test_attention_matches_library_sdpa():
    import torch
    rng = np.random.default_rng(11)
    H, nq, T, D = 3, 5, 37, 16
    q = rng.standard_normal((H, nq, D))
    K = rng.standard_normal((H, T, D))
    V = rng.standard_normal((H, T, D))
    for scale in (1.0 / np.sqrt(D), 0.7):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V), scale=scale).numpy()
        assert np.allclose(jolt.attention(q, K, V, scale), ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(12)
    H, nq, T, D = 2, 3, 9, 8
    q = rng.standard_normal((H, nq, D))
    V = rng.standard_normal((H, T, D))
    # every key equal: uniform weights, the mean value row
    K = np.repeat(rng.standard_normal((H, 1, D)), T, axis=1)
    assert np.allclose(jolt.attention(q, K, V, 0.5), np.repeat(V.mean(axis=1, keepdims=True),
                                                               nq, axis=1), atol=1e-14)
    # one token: its value row, whatever the score
    assert np.allclose(jolt.attention(q, K[:, :1], V[:, :1], 3.0),
                       np.repeat(V[:, :1], nq, axis=1), atol=1e-14)
    # a key aligned with the query and a large scale: that token's value row
    K = rng.standard_normal((H, T, D)) * 0.01
    K[:, 4] = q[:, 0] * 10.0
    out = jolt.attention(q[:, :1], K, V, 50.0)
    assert np.allclose(out[:, 0], V[:, 4], atol=1e-12)
    # tokens permuted jointly in K and V: the same output
    K = rng.standard_normal((H, T, D))
    perm = rng.permutation(T)
    assert np.allclose(jolt.attention(q, K, V, 0.3), jolt.attention(q, K[:, perm], V[:, perm], 0.3),
                       atol=1e-13)


@pytest.mark.parametrize("rT,rd,b", [(5, 4, 4), (16, 32, 0), (16, 8, 8), (5, 32, 2)])
def test_random_blob_sections_read_back(rT, rd, b):
    rng = np.random.default_rng(rT * 100 + rd + b)
    H, T, D = 3, 16, 32
    signs = np.where(rng.random(D) < 0.5, -1, 1).astype(np.int8)
    blob = jolt.random_blob(rng, H, T, D, rT, rd, b, signs)
    hd = jolt.parse_header(blob)
    assert (hd["H"], hd["T"], hd["D"], hd["rT"], hd["rd"], hd["b"]) == (H, T, D, rT, rd, b)
    assert np.array_equal(hd["signs"], signs)
    assert hd["bytes"] == len(blob) == jolt.blob_layout(H, T, D, rT, rd, b, D)["bytes"]
    X = jolt.decode_unit(blob)
    assert X.shape == (H, T, D) and np.all(np.isfinite(X))


def test_attend_group_full_rank_no_residual_is_attention_on_fp16_tensors():
    """Full ranks and b = 0 store G = X in fp16, so attention over the blobs
    is attention over the fp16-rounded K and V."""
    rng = np.random.default_rng(13)
    Kx = rng.standard_normal((2, 16, 32))
    Vx = rng.standard_normal((2, 16, 32))
    signs = np.ones(32, dtype=np.int8)
    blobs = []
    for X in (Kx, Vx):
        fac = jolt.factorize(X, (jolt.FULL,), (jolt.FULL,))
        blobs.append(jolt.encode_unit(X, fac, signs, 16, 32, 0, 32))
    q = rng.standard_normal((2, 3, 32))
    ref = jolt.attention(q, jolt.f16(Kx), jolt.f16(Vx), 0.25)
    assert np.allclose(jolt.attend_group(q, blobs[0], blobs[1], 0.25), ref, atol=1e-13)


# ---------------------------------------------------------------- admission
def test_cholesky_solve_drop_matches_library_solve():
    rng = np.random.default_rng(41)
    for n in (1, 5, 17):
        A = rng.standard_normal((n, n + 3))
        M = A @ A.T
        rhs = rng.standard_normal((4, n))
        ref = np.linalg.solve(M, rhs.T).T
        assert np.allclose(jolt.cholesky_solve_drop(M, rhs), ref, rtol=1e-10, atol=1e-12)


def test_cholesky_solve_drop_zero_pivots():
    M = np.diag([4.0, 0.0, 2.0, 0.0])
    rhs = np.array([[8.0, 5.0, -2.0, 7.0]])
    assert np.allclose(jolt.cholesky_solve_drop(M, rhs), np.array([[2.0, 0.0, -1.0, 0.0]]),
                       rtol=0, atol=1e-15)
    assert np.array_equal(jolt.cholesky_solve_drop(np.zeros((3, 3)), np.ones((1, 3))),
                          np.zeros((1, 3)))


def test_fold_in_returns_the_tokens_own_row():
    """With the unrounded factors of an exact ST-HOSVD (U_T the leading
    eigenvectors of the token Gram, G = U_T^T Y), the least-squares
    coordinates of any existing token are its row of U_T."""
    w = kvgen.custom_workload("tiny", H=4, T=40, D=32)
    X = kvgen.make_unit_f64(w, 0)
    fac = jolt.factorize(X, (8, jolt.FULL), (8, jolt.FULL))
    for rd in fac.rd_list:
        Y, UT, G = fac.Y[rd], fac.UT[rd][:, :8], fac.G[rd][:, :8, :]
        u = jolt.fold_in(Y[:, 3:9, :], G)
        assert np.allclose(u, UT[3:9], atol=1e-9), rd


def _admit_case(rT, rd, b, T=24, tau=10, seed=0):
    rng = np.random.default_rng(seed)
    w = kvgen.custom_workload("tiny", H=3, T=T + tau, D=32)
    X = kvgen.make_unit_f64(w, 1)
    signs = kvgen.make_signs(w, 1)
    fac = jolt.factorize(X[:, :T], (rT,), (rd,))
    blob = jolt.encode_unit(X[:, :T], fac, signs, fac.rT_list[0], fac.rd_list[0], b, 32)
    return blob, X[:, T:], rng


@pytest.mark.parametrize("rT,rd,b", [(6, 8, 4), (jolt.FULL, 8, 2), (6, jolt.FULL, 8),
                                     (jolt.FULL, jolt.FULL, 4), (4, 4, 0)])
def test_admit_keeps_old_tokens_and_bounds_new_error(rT, rd, b):
    blob, Xn, _ = _admit_case(rT, rd, b)
    out = jolt.admit_unit(blob, Xn)
    hd, ho = jolt.parse_header(blob), jolt.parse_header(out)
    T, tau = hd["T"], Xn.shape[1]
    assert ho["T"] == T + tau and ho["rd"] == hd["rd"] and ho["b"] == hd["b"]
    assert ho["rT"] == (T + tau if hd["rT"] == T else hd["rT"])
    assert np.array_equal(ho["signs"], hd["signs"])
    old, new = jolt.decode_unit(blob), jolt.decode_unit(out)
    assert np.array_equal(new[:, :T], old)
    if b > 0:
        # every new row's rotated error is within half its quantization step
        Q = jolt.rotation_matrix(ho["signs"])
        s = np.frombuffer(out, dtype=np.float16, count=3 * (T + tau),
                          offset=ho["scale"]).astype(np.float64).reshape(3, T + tau)[:, T:]
        err = np.abs((new[:, T:] - Xn).reshape(-1, 32) @ Q.T)
        assert np.all(err <= 0.5 * s.reshape(-1, 1) * (1 + 1e-9) + 1e-12)


def test_admit_whole_modes_no_residual_is_fp16_of_the_block():
    blob, Xn, _ = _admit_case(jolt.FULL, jolt.FULL, 0)
    out = jolt.admit_unit(blob, Xn)
    assert np.array_equal(jolt.decode_unit(out)[:, 24:], jolt.f16(Xn))


def test_admit_tokens_in_the_factor_span_have_zero_residual():
    """r_d = D (Y = X): a block u* G16 in the span of the stored core gets
    back u* as its U_T rows and a zero residual (zero scales)."""
    blob, Xn, rng = _admit_case(6, jolt.FULL, 4)
    hd = jolt.parse_header(blob)
    G = np.frombuffer(blob, dtype=np.float16, count=3 * 6 * 32, offset=hd["G"]).astype(
        np.float64).reshape(3, 6, 32)
    u_star = jolt.f16(rng.standard_normal((5, 6)) * 0.1)
    X_span = jolt.reconstruct(u_star, G, None)
    out = jolt.admit_unit(blob, X_span)
    ho = jolt.parse_header(out)
    UT = np.frombuffer(out, dtype=np.float16, count=(24 + 5) * 6, offset=ho["UT"]).astype(
        np.float64).reshape(29, 6)
    assert np.array_equal(UT[24:], u_star)
    s = np.frombuffer(out, dtype=np.float16, count=3 * 29, offset=ho["scale"]).reshape(3, 29)
    assert np.all(s[:, 24:] == 0)


@pytest.mark.parametrize("rT,rd,b", [(6, 8, 4), (jolt.FULL, 8, 2)])
def test_admit_two_blocks_equals_one_block(rT, rd, b):
    blob, Xn, _ = _admit_case(rT, rd, b)
    one = jolt.admit_unit(blob, Xn)
    two = jolt.admit_unit(jolt.admit_unit(blob, Xn[:, :4]), Xn[:, 4:])
    assert one == two
