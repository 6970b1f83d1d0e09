"""The main path at full size on the four large configurations, in the
launch the bench uses (all units of a configuration in one batch, the
bisection then the greedy swaps):

  mistral_t1024  8 groups x {K,V} of [32, 1024, 128], exact, 2x budget
  mistral_t2048  8 groups x {K,V} of [32, 2048, 128], exact, 3x budget
  llama_t1024    10 groups x {K,V} of [160, 1024, 128], exact, 2x budget
  flash_t4096    8 groups x {K,V} of [32, 4096, 128], randomized, 2x budget

The oracle cannot run its exhaustive grid on 1024-4096-token units in
seconds, so each configuration checks what it can compute exactly:

  * the cost table, bit for bit (oracle cost_table);
  * the allocation and the greedy swaps, bit for bit, on the GPU's tables
    (oracle allocate / refine_greedy);
  * every b = 0 entry of one sampled unit against its ST-HOSVD tail
    ||X||^2 - ||G(r_T, r_d)||^2, at the path's tolerance (fp16 storage of
    the factors moves these values by ~1e-7 relative): exact modes take the
    token-Gram eigenvalues (numpy eigvalsh), the randomized mode the
    oracle's own FlashJoLT factors on the same sketch;
  * the chosen candidate's table entry against the distortion of what the
    GPU's decoder rebuilds from the blob (fp32 and bf16 output), every unit;
  * the codes of up to four units against the oracle's quantizer on the
    blob's stored factors (the bar of the small parity tests);
  * b > 0 and b = 0 table entries of two units (one K, one V) on five rank
    pairs spread over the grid, every bit width, against the oracle's
    distortion of the same candidate: each candidate is serialized in
    turn, and the oracle rebuilds X~ from the blob's fp16 factors, quantizes
    the rotated residual with its own quantizer and measures D in f64
    (the fused sweep's scoring against the definition, at full size);
  * the modeled table (unrounded factors) of the sampled unit against the
    same tails.

The oracle's own Jacobi does not finish a 1024 x 1024 token Gram in ten
minutes, so the exact token spectra at full size come from LAPACK
(numpy eigvalsh); the Jacobi is pinned against it at small sizes.
"""
import numpy as np
import pytest

import kvgen
from oracle import jolt as oj
from partial_tucker_rotated_st_b300.codec import config_for as codec_cfg
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-6
BIG = ["mistral_t1024", "mistral_t2048", "llama_t1024", "flash_t4096"]


def _b0_reference(w, x, sk):
    """[n_rT][n_rd] of ||X - X~||^2 / ||X||^2 for the unrounded factors."""
    xn = float(np.sum(x * x))
    rT = [oj.resolve(v, w.T) for v in w.rT]
    rd = [oj.resolve(v, w.D) for v in w.rd]
    out = np.zeros((len(rT), len(rd)))
    if w.token_mode == "randomized":
        fac = oj.factorize(x, w.rT, w.rd, "randomized", sk, w.power_iters)
        for j, r_d in enumerate(rd):
            ny = float(np.sum(fac.Y[r_d] ** 2))
            g2 = np.sum(fac.G[r_d] ** 2, axis=(0, 2))      # per token rank
            for i, r_T in enumerate(rT):
                cap = ny if r_T == w.T else float(np.sum(g2[:r_T]))
                out[i, j] = max(xn - cap, 0.0) / xn
        return out
    _, V = oj.feature_mode(x)
    for j, r_d in enumerate(rd):
        Y = x if r_d == w.D else np.einsum("htd,dj->htj", x, V[:, :r_d])
        A = oj.token_unfolding(Y)
        mu = np.linalg.eigvalsh(A @ A.T)[::-1]
        for i, r_T in enumerate(rT):
            cap = float(np.sum(mu[:r_T])) if r_T < w.T else float(np.sum(Y * Y))
            out[i, j] = max(xn - cap, 0.0) / xn
    return out


def _rank_pairs(nT, nd):
    """Five (iT, id) cells spread over the grid: the corners and the middle."""
    out = []
    for c in [(0, 0), (nT - 1, nd - 1), (nT // 2, nd // 2), (0, nd - 1), (nT - 1, 0),
              (1, nd - 2), (nT - 2, 1)]:
        if c not in out and 0 <= c[0] < nT and 0 <= c[1] < nd:
            out.append(c)
    return out[:5]


def _check_candidates(w, r, units=(2, 3)):
    """Table entries of every bit width on five rank pairs against the
    oracle's distortion of the candidate's own stored factors (the factors of
    a rank pair are the same for every b, so one blob per pair serves all)."""
    import torch
    enc, X, S, _ = r.dev
    nT, nd, nb = len(w.rT), len(w.rd), len(w.bits)
    ib_top = int(np.argmax(w.bits))
    for iT, id_ in _rank_pairs(nT, nd):
        c_top = (iT * nd + id_) * nb + ib_top
        desc = enc.serialize(X, S, [c_top] * len(r.units))
        torch.cuda.synchronize()
        for u in units:
            blob = enc.blob[u, :desc[u].bytes].cpu().numpy().tobytes()
            hd = oj.parse_header(blob)
            Xt = _stored_xtilde(blob, hd)
            Q = oj.rotation_matrix(hd["signs"])
            x = r.X64[u]
            for ib, b in enumerate(w.bits):
                c = (iT * nd + id_) * nb + ib
                ref = oj.distortion(x, oj.candidate_xhat(x, Xt, Q, b))
                got = float(r.dist[u, c])
                assert abs(got - ref) <= max(REL * ref, ABS), \
                    (u, c, (hd["rT"], hd["rd"], b), got, ref)


def _stored_xtilde(blob, hd):
    H, T, D, rT, rd = hd["H"], hd["T"], hd["D"], hd["rT"], hd["rd"]

    def arr(off, n, shape):
        return np.frombuffer(blob, np.float16, n, off).astype(np.float64).reshape(shape)

    UT = None if hd["flags"] & 1 else arr(hd["UT"], T * rT, (T, rT))
    Ud = None if hd["flags"] & 2 else arr(hd["Ud"], D * rd, (D, rd))
    G = arr(hd["G"], H * rT * rd, (H, rT, rd))
    return oj.reconstruct(UT, G, Ud)


@pytest.mark.parametrize("name", BIG)
def test_full_size_config(name):
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    from tests.test_gpu_parity import check_codes_against_oracle
    w = kvgen.WORKLOADS[name]
    r = gh.run(w, refine=True, keep=True)
    U = w.n_units
    assert r.status == 0
    # cost table
    rT = [oj.resolve(x, w.T) for x in w.rT]
    rd = [oj.resolve(x, w.D) for x in w.rd]
    ref = oj.cost_table(w.H, w.T, w.D, rT, rd, w.bits, w.block).reshape(-1)
    for u in range(U):
        assert np.array_equal(r.cost[u], ref)
    # bisection and greedy swaps on the GPU's tables
    z, lam, st = oj.allocate(r.dist, r.cost, w.budget_bytes, 256)
    assert st == oj.ALLOC_OK and lam == r.lam
    zr, _ = oj.refine_greedy(r.dist, r.cost, w.budget_bytes, np.array(z))
    assert list(zr) == list(r.choice)
    assert sum(int(r.cost[u, zr[u]]) for u in range(U)) <= w.budget_bytes
    # b = 0 entries of a sampled unit (a K unit with its outlier channels)
    u = 2
    sk = None if r.sketch is None else r.sketch[u].astype(np.float64)
    b0 = _b0_reference(w, r.X64[u], sk)
    d = r.dist[u].reshape(len(rT), len(rd), len(w.bits))[:, :, w.bits.index(0)]
    bad = np.abs(d - b0) > np.maximum(REL * b0, ABS)
    assert not bad.any(), [(rT[i], rd[j], d[i, j], b0[i, j]) for i, j in np.argwhere(bad)]
    # the modeled table of the same unit: eps^2(b) times the same tails
    enc = r.dev[0]
    eps2 = [1.0 if b == 0 else 4.0 ** (-b) for b in w.bits]
    md = torch.zeros(U, enc.ncand, dtype=torch.float64, device="cuda")
    J.jolt_model_candidates(codec_cfg(w), U, enc.ws, eps2, md)
    torch.cuda.synchronize()
    md = md[u].cpu().numpy().reshape(len(rT), len(rd), len(w.bits))
    for ib in range(len(w.bits)):
        ref_m = eps2[ib] * b0
        bad = np.abs(md[:, :, ib] - ref_m) > np.maximum(REL * ref_m, ABS)
        assert not bad.any(), [(rT[i], rd[j], w.bits[ib], md[i, j, ib], ref_m[i, j])
                               for i, j in np.argwhere(bad)]
    # b > 0 (and b = 0) cells of two units against the oracle's distortion
    _check_candidates(w, r)
    # the chosen candidates are what decodes (fp32 and bf16 output)
    for u in range(U):
        x = r.X64[u]
        xx = float(np.sum(x * x))
        e = x - r.xhat32[u]
        got = float(np.sum(e * e)) / xx
        c = int(r.choice[u])
        assert abs(r.dist[u, c] - got) <= max(1e-4 * got, 1e-7), (u, r.dist[u, c], got)
        x16 = kvgen.bf16_to_f32(r.xhat16[u]).astype(np.float64)
        assert np.all(np.abs(x16 - r.xhat32[u]) <= 2.0 ** -8 * np.abs(r.xhat32[u]) + 1e-30)
    # codes of up to four units with b > 0
    bad = tot = done = 0
    for u in range(U):
        if done == 4:
            break
        if oj.parse_header(r.blobs[u])["b"] == 0:
            continue
        nbad, n = check_codes_against_oracle(r.X64[u], r.blobs[u], w.D)
        bad, tot, done = bad + nbad, tot + n, done + 1
    assert bad <= max(1e-4 * tot, 8), (bad, tot)
