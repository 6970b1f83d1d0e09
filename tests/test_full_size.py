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
    blob's stored factors (the bar of the small parity tests).
"""
import numpy as np
import pytest

import kvgen
from oracle import jolt as oj
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


@pytest.mark.parametrize("name", BIG)
def test_full_size_config(name):
    from tests.test_gpu_parity import check_codes_against_oracle
    w = kvgen.WORKLOADS[name]
    r = gh.run(w, refine=True)
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
