"""Pins for the FP64 oracle, each against something other than the oracle.

The equations are those of "Writing Speed-of-Light Attention Backward Kernel
for 5090 in CUDA", section "Mathematical Formulation" (forward and backward)
and Appendix B (softmax backward).  Each pin below is chosen so that a
plausible slip in the oracle (a dropped scale, an off-by-one causal mask, a
wrong LSE base, a missing D term, a transposed operand) fails at least one of
them; ``test_pins_catch_planted_mistakes`` plants such slips in a copy of the
oracle source and checks exactly that.
"""
import itertools
import math
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attn_fwd(q, k, v, scale, causal)
    return float(np.sum(dout * o))


# ---------------------------------------------------------------- finite differences
@pytest.mark.parametrize("N,d,causal", [(5, 3, True), (5, 3, False), (8, 4, True), (7, 4, False)])
def test_gradients_match_central_differences(N, d, causal):
    """dQ, dK, dV equal the central differences of the scalar loss sum(dO o O)."""
    BH = 2
    scale = 0.7  # deliberately not 1/sqrt(d): the scale must enter exactly where it should
    q, k, v, dout = (_rand((BH, N, d), s) for s in (1, 2, 3, 4))
    g = oracle.attn_bwd(q, k, v, dout, scale, causal)
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in itertools.product(*(range(s) for s in x.shape)):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            argm = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            fd[idx] = (_loss(*args, dout, scale, causal) - _loss(*argm, dout, scale, causal)) / (2 * h)
        err = np.max(np.abs(fd - g[name])) / max(1e-12, np.max(np.abs(g[name])))
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------- Q = 0 closed form
@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_closed_form(causal):
    """Q = 0: S = M, so P is uniform over unmasked keys."""
    N, d, scale = 9, 5, 0.35
    q = np.zeros((1, N, d))
    k, v, dout = _rand((1, N, d), 11), _rand((1, N, d), 12), _rand((1, N, d), 13)
    g = oracle.attn_bwd(q, k, v, dout, scale, causal)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal)
    i = np.arange(N)
    if causal:
        o_ref = np.cumsum(v[0], axis=0) / (i + 1)[:, None]          # mean of V over the prefix
        lse_ref = np.log(i + 1.0)                                    # log(i+1), 0-based i
        dv_ref = np.array([np.sum(dout[0, j:] / (i[j:] + 1.0)[:, None], axis=0) for j in range(N)])
    else:
        o_ref = np.broadcast_to(v[0].mean(axis=0), (N, d))
        lse_ref = np.full(N, np.log(N))
        dv_ref = np.broadcast_to(dout[0].sum(axis=0) / N, (N, d))
    np.testing.assert_allclose(o[0], o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], lse_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dv"][0], dv_ref, rtol=0, atol=1e-12)
    assert np.all(g["dk"] == 0.0)  # dK = scale * dS^T Q with Q = 0, exactly


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [True, False])
def test_row_invariants(causal):
    N, d, scale = 12, 6, 0.5
    q, k, v, dout = (_rand((N, d), s) for s in (21, 22, 23, 24))
    P, dS = oracle.attn_probs(q, k, v, scale, causal, dout)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)      # rows of P sum to 1
    np.testing.assert_allclose(dS.sum(axis=1), 0.0, rtol=0, atol=1e-13)     # rows of dS sum to 0
    if causal:
        assert np.all(P[np.triu_indices(N, 1)] == 0.0)                       # masked entries exactly 0
    g = oracle.attn_bwd(q[None], k[None], v[None], dout[None], scale, causal)
    np.testing.assert_allclose(g["dk"][0].sum(axis=0), 0.0, rtol=0, atol=1e-12)  # sum_j dK_j = 0
    # D two ways: rowsum(dO o O) == rowsum(P o dP)
    dP = dout @ v.T
    np.testing.assert_allclose(g["delta"][0], np.sum(P * dP, axis=1), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- special cases
def test_single_key():
    """N = 1: O = V, dQ = dK = 0, dV = dO, L = scale q.k."""
    d, scale = 7, 0.9
    q, k, v, dout = (_rand((1, 1, d), s) for s in (31, 32, 33, 34))
    for causal in (True, False):
        g = oracle.attn_bwd(q, k, v, dout, scale, causal)
        np.testing.assert_allclose(g["o"], v, atol=1e-15)
        np.testing.assert_allclose(g["lse"][0, 0], scale * float(q[0, 0] @ k[0, 0]), atol=1e-14)
        np.testing.assert_allclose(g["dq"], 0.0, atol=1e-15)
        np.testing.assert_allclose(g["dk"], 0.0, atol=1e-15)
        np.testing.assert_allclose(g["dv"], dout, atol=1e-15)


def test_causal_first_row():
    N, d, scale = 6, 4, 0.8
    q, k, v = (_rand((1, N, d), s) for s in (41, 42, 43))
    o, lse = oracle.attn_fwd(q, k, v, scale, True)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], scale * float(q[0, 0] @ k[0, 0]), atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_key_shift_invariance(causal):
    """K -> K + 1 c^T leaves O, dQ, dV unchanged and shifts L_i by scale q_i.c."""
    N, d, scale = 10, 5, 0.6
    q, k, v, dout = (_rand((1, N, d), s) for s in (51, 52, 53, 54))
    c = _rand((d,), 55)
    a = oracle.attn_bwd(q, k, v, dout, scale, causal)
    b = oracle.attn_bwd(q, k + c, v, dout, scale, causal)
    np.testing.assert_allclose(b["o"], a["o"], atol=1e-12)
    np.testing.assert_allclose(b["dq"], a["dq"], atol=1e-12)
    np.testing.assert_allclose(b["dv"], a["dv"], atol=1e-12)
    np.testing.assert_allclose(b["lse"][0], a["lse"][0] + scale * (q[0] @ c), atol=1e-12)


def test_key_permutation_invariance_noncausal():
    N, d, scale = 11, 4, 0.7
    q, k, v = (_rand((1, N, d), s) for s in (61, 62, 63))
    perm = np.random.default_rng(64).permutation(N)
    o1, l1 = oracle.attn_fwd(q, k, v, scale, False)
    o2, l2 = oracle.attn_fwd(q, k[:, perm], v[:, perm], scale, False)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)


# ---------------------------------------------------------------- library routine
@pytest.mark.parametrize("causal", [True, False])
def test_matches_scipy_softmax(causal):
    """Dense softmax and logsumexp from scipy on the whole score matrix."""
    from scipy.special import logsumexp, softmax
    N, d, scale = 33, 8, 1 / math.sqrt(8)
    q, k, v = (_rand((N, d), s) for s in (71, 72, 73))
    S = scale * q @ k.T
    if causal:
        S = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, S)
    o, lse = oracle.attn_fwd(q[None], k[None], v[None], scale, causal)
    np.testing.assert_allclose(o[0], softmax(S, axis=1) @ v, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], logsumexp(S, axis=1), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- brute force
def _brute(q, k, v, dout, scale, causal):
    """Untiled scalar loops straight from the equations (pure Python)."""
    N, d = len(q), len(q[0])
    S = [[scale * sum(q[i][c] * k[j][c] for c in range(d)) + (-math.inf if causal and j > i else 0.0)
          for j in range(N)] for i in range(N)]
    L = [math.log(sum(math.exp(S[i][j]) for j in range(N))) for i in range(N)]
    P = [[math.exp(S[i][j] - L[i]) for j in range(N)] for i in range(N)]
    O = [[sum(P[i][j] * v[j][c] for j in range(N)) for c in range(d)] for i in range(N)]
    D = [sum(dout[i][c] * O[i][c] for c in range(d)) for i in range(N)]
    dP = [[sum(dout[i][c] * v[j][c] for c in range(d)) for j in range(N)] for i in range(N)]
    dS = [[P[i][j] * (dP[i][j] - D[i]) for j in range(N)] for i in range(N)]
    dQ = [[scale * sum(dS[i][j] * k[j][c] for j in range(N)) for c in range(d)] for i in range(N)]
    dK = [[scale * sum(dS[i][j] * q[i][c] for i in range(N)) for c in range(d)] for j in range(N)]
    dV = [[sum(P[i][j] * dout[i][c] for i in range(N)) for c in range(d)] for j in range(N)]
    return O, L, dQ, dK, dV


@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_tiny(causal):
    N, d, scale = 6, 3, 0.45
    q, k, v, dout = (_rand((N, d), s) for s in (81, 82, 83, 84))
    O, L, dQ, dK, dV = _brute(q.tolist(), k.tolist(), v.tolist(), dout.tolist(), scale, causal)
    g = oracle.attn_bwd(q[None], k[None], v[None], dout[None], scale, causal)
    for a, b in ((g["o"][0], O), (g["lse"][0], L), (g["dq"][0], dQ), (g["dk"][0], dK), (g["dv"][0], dV)):
        np.testing.assert_allclose(a, np.array(b), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- entry points agree
@pytest.mark.parametrize("causal", [True, False])
def test_row_entry_point_matches_whole_head(causal):
    N, d, scale = 40, 8, 0.3
    q, k, v, dout = (_rand((N, d), s) for s in (91, 92, 93, 94))
    g = oracle.attn_bwd(q[None], k[None], v[None], dout[None], scale, causal)
    rows = [0, 1, 17, 39]
    o, lse, dq = oracle.attn_rows(q, k, v, rows, scale, causal, dout=dout)
    np.testing.assert_allclose(o, g["o"][0][rows], atol=1e-14)
    np.testing.assert_allclose(lse, g["lse"][0][rows], atol=1e-14)
    np.testing.assert_allclose(dq, g["dq"][0][rows], atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_rowset_parts_sum_to_whole_head(causal):
    """Splitting the query rows into sets and adding their dK/dV parts gives
    the whole-head dK/dV; dQ rows match."""
    N, d, scale = 24, 5, 0.4
    q, k, v, dout = (_rand((N, d), s) for s in (95, 96, 97, 98))
    g = oracle.attn_bwd(q[None], k[None], v[None], dout[None], scale, causal)
    dk = np.zeros((N, d)); dv = np.zeros((N, d))
    for rows in (list(range(0, N, 3)), list(range(1, N, 3)), list(range(2, N, 3))):
        dq_r, dk_p, dv_p = oracle.attn_bwd_rowset(q, k, v, dout, rows, scale, causal)
        np.testing.assert_allclose(dq_r, g["dq"][0][rows], atol=1e-14)
        dk += dk_p; dv += dv_p
    np.testing.assert_allclose(dk, g["dk"][0], atol=1e-13)
    np.testing.assert_allclose(dv, g["dv"][0], atol=1e-13)


def test_rejects_bad_rows():
    q = np.zeros((4, 2))
    with pytest.raises(RuntimeError):
        oracle.attn_rows(q, q, q, [4], 1.0, False)


# ---------------------------------------------------------------- planted mistakes
MUTATIONS = {
    "dK loses its scale": ("dkh[j * d + c] += scale * ds[j] * qh[i * d + c]", "dkh[j * d + c] += ds[j] * qh[i * d + c]"),
    "mask keeps one key too many": ("(causal && j > i)", "(causal && j > i + 1)"),
    "mask drops the diagonal": ("(causal && j > i)", "(causal && j >= i && i > 0)"),
    "LSE in base 2": ("return m + log(acc);", "return m + log2(acc);"),
    "D term dropped": ("ds[j] = p[j] * (dp - D);", "ds[j] = p[j] * dp;"),
    "dQ uses V for K": ("dq_i[c] += ds[j] * k[j * d + c];", "dq_i[c] += ds[j] * v[j * d + c];"),
    "dV uses dS for P": ("dvh[j * d + c] += p[j] * doh[i * d + c];", "dvh[j * d + c] += ds[j] * doh[i * d + c];"),
}

_PINS = [
    lambda: test_gradients_match_central_differences(5, 3, True),
    lambda: test_gradients_match_central_differences(7, 4, False),
    lambda: test_zero_query_closed_form(True),
    lambda: test_zero_query_closed_form(False),
    lambda: test_row_invariants(True),
    lambda: test_matches_scipy_softmax(True),
    lambda: test_brute_force_tiny(True),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name):
    """Each planted slip in a copy of the oracle fails at least one pin."""
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, name
    tmp = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        path = os.path.join(tmp, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load_library(oracle.build(force=True, src=path, out=os.path.join(tmp, "libmut.so")))
        prev = oracle.use_library(lib)
        try:
            failures = 0
            for pin in _PINS:
                try:
                    pin()
                except AssertionError:
                    failures += 1
            assert failures > 0, f"no pin caught: {name}"
        finally:
            oracle.use_library(prev)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
