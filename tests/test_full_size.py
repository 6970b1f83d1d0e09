"""The main path at the bench's size and launch configuration: mistral_t1024,
16 units of [32, 1024, 128] bf16 in one batch, exact token mode, the
bisection then the greedy swaps.  The oracle cannot factor 1024-token units
in seconds, so this file checks what it can compute exactly at this size:

  * the cost table, bit for bit (oracle cost_table);
  * the allocation and the greedy swaps, bit for bit, on the GPU's tables
    (oracle allocate / refine_greedy);
  * every b = 0 entry of two sampled units against the exact ST-HOSVD tail
    ||X||^2 - sum_{j < r_T} mu_j(r_d) of that unit (oracle feature mode,
    token-Gram eigenvalues by numpy's eigvalsh), at the path's tolerance
    (fp16 storage of the factors moves these values by ~1e-7 relative);
  * the chosen candidate's table entry against the distortion of what the
    GPU's decoder rebuilds from the blob, for every unit;
  * the codes of four units against the oracle's quantizer on the blob's
    stored factors (the same bar as the small parity tests).
"""
import numpy as np
import pytest

import kvgen
from oracle import jolt as oj
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

REL, ABS = 1e-3, 1e-6
W = kvgen.WORKLOADS["mistral_t1024"]
_RUN = {}


def full_run():
    if "r" not in _RUN:
        _RUN["r"] = gh.run(W, refine=True)
    return _RUN["r"]


def test_full_size_status_and_cost_table():
    r = full_run()
    assert r.status == 0
    rT = [oj.resolve(x, W.T) for x in W.rT]
    rd = [oj.resolve(x, W.D) for x in W.rd]
    ref = oj.cost_table(W.H, W.T, W.D, rT, rd, W.bits, W.block).reshape(-1)
    for u in range(W.n_units):
        assert np.array_equal(r.cost[u], ref)


def test_full_size_allocation_and_refinement_bit_exact():
    r = full_run()
    z, lam, st = oj.allocate(r.dist, r.cost, W.budget_bytes, 256)
    assert st == oj.ALLOC_OK and lam == r.lam
    zr, _ = oj.refine_greedy(r.dist, r.cost, W.budget_bytes, np.array(z))
    assert list(zr) == list(r.choice)
    assert sum(int(r.cost[u, zr[u]]) for u in range(W.n_units)) <= W.budget_bytes


@pytest.mark.parametrize("u", [0, 5])
def test_full_size_b0_distortions_are_the_hosvd_tails(u):
    r = full_run()
    x = r.X64[u]
    xn = float(np.sum(x * x))
    _, V = oj.feature_mode(x)
    rT = [oj.resolve(v, W.T) for v in W.rT]
    rd = [oj.resolve(v, W.D) for v in W.rd]
    d = r.dist[u].reshape(len(rT), len(rd), len(W.bits))
    for j, r_d in enumerate(rd):
        Y = x if r_d == W.D else np.einsum("htd,dj->htj", x, V[:, :r_d])
        A = oj.token_unfolding(Y)
        mu = np.linalg.eigvalsh(A @ A.T)[::-1]
        for i, r_T in enumerate(rT):
            cap = float(np.sum(mu[:r_T])) if r_T < W.T else float(np.sum(Y * Y))
            ref = max(xn - cap, 0.0) / xn
            got = d[i, j, W.bits.index(0)]
            assert abs(got - ref) <= max(REL * ref, ABS), (r_T, r_d, got, ref)


def test_full_size_chosen_candidate_is_what_decodes():
    r = full_run()
    for u in range(W.n_units):
        x = r.X64[u]
        e = x - r.xhat32[u]
        got = float(np.sum(e * e) / np.sum(x * x))
        c = int(r.choice[u])
        assert abs(r.dist[u, c] - got) <= max(1e-4 * got, 1e-7), (u, r.dist[u, c], got)


def test_full_size_codes_match_oracle_quantizer():
    from tests.test_gpu_parity import check_codes_against_oracle
    r = full_run()
    bad = tot = 0
    for u in range(W.n_units):
        if oj.parse_header(r.blobs[u])["b"] == 0:
            continue
        nbad, n = check_codes_against_oracle(r.X64[u], r.blobs[u], W.D)
        bad, tot = bad + nbad, tot + n
        if tot > 4 * W.elems_per_unit:
            break
    assert tot > 0 and bad <= max(1e-4 * tot, 8), (bad, tot)
