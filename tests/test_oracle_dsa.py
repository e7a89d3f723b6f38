"""Pins for the FP64 sparse top-k attention oracle (``oracle/dsa.py``), each against
something other than that oracle: finite differences of a scalar loss, the dense
oracle (a separate C implementation) when every row lists all keys in order, the
q = 0 closed form with a sink, invariance under reordering a row's index list,
and sink -> -inf equal to no sink.  ``test_pins_catch_planted_mistakes`` plants
plausible slips in a copy of the oracle source and checks that each one fails at
least one pin.
"""
import importlib.util
import itertools
import math
import os
import sys
import types

import numpy as np
import pytest

import oracle
from oracle import dsa as dsa_mod

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa.py")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _tiny_case(sink=True):
    """s_q = 5 queries, 7 keys, 2 heads, d_qk = 5, d_v = 3; lists with a padding
    entry, an out-of-range index, a duplicate, keys after the query (masked when
    causal), a shortened row and an empty row."""
    s_q, s_kv, H, d_qk, d_v = 5, 7, 2, 5, 3
    q = _rand((s_q, H, d_qk), 1)
    kv = _rand((s_kv, d_qk), 2)
    do = _rand((s_q, H, d_v), 3)
    snk = _rand((H,), 4) if sink else None
    idx = np.array([[0, 3, -1, 5, 1],
                    [1, 1, 0, 6, 2],
                    [2, 9, 0, 1, 4],
                    [3, 0, 2, 6, 5],
                    [4, 2, 1, 0, 3]], dtype=np.int32)
    lens = np.array([5, 4, 5, 0, 3], dtype=np.int32)
    return dict(q=q, kv=kv, do=do, sink=snk, idx=idx, lens=lens, d_v=d_v)


# --------------------------------------------------------------------------- pins
def pin_finite_differences(m, causal, sink=True):
    """dq, dkv, dsink equal the central differences of sum(dO o O) through m.dsa_fwd."""
    c = _tiny_case(sink)
    scale = 0.7

    def loss(q, kv, snk):
        o, _ = m.dsa_fwd(q, kv, snk, c["idx"], c["lens"], scale, causal, c["d_v"])
        return float(np.sum(c["do"] * o))

    o, lse = m.dsa_fwd(c["q"], c["kv"], c["sink"], c["idx"], c["lens"], scale, causal, c["d_v"])
    g = m.dsa_bwd(c["q"], c["kv"], o, c["do"], lse, c["sink"], c["idx"], c["lens"], scale, causal, c["d_v"])
    h = 1e-6
    targets = [("dq", "q"), ("dkv", "kv")] + ([("dsink", "sink")] if sink else [])
    for gname, xname in targets:
        x = c[xname]
        fd = np.zeros_like(x)
        for ix in itertools.product(*(range(s) for s in x.shape)):
            args_p = {k: c[k].copy() if c[k] is not None else None for k in ("q", "kv", "sink")}
            args_m = {k: c[k].copy() if c[k] is not None else None for k in ("q", "kv", "sink")}
            args_p[xname][ix] += h
            args_m[xname][ix] -= h
            fd[ix] = (loss(args_p["q"], args_p["kv"], args_p["sink"]) -
                      loss(args_m["q"], args_m["kv"], args_m["sink"])) / (2 * h)
        ref = g[gname]
        if ref is None:
            return False
        err = np.max(np.abs(fd - ref)) / max(1e-12, np.max(np.abs(fd)))
        if not err < 1e-6:
            return False
    return True


def pin_dense_reduction(m, causal, d_qk, d_v):
    """Every row lists all keys 0..N-1 in order, no sink: the dense attention of
    each head with K = kv and V = kv[:, :d_v] (the dense C oracle, V and dO padded
    with zero columns to d_qk).  dkv = sum over heads of dK + dV."""
    N, H, scale = 6, 3, 0.45
    q = _rand((N, H, d_qk), 21)
    kv = _rand((N, d_qk), 22)
    do = _rand((N, H, d_v), 23)
    idx = np.tile(np.arange(N, dtype=np.int32), (N, 1))
    o, lse = m.dsa_fwd(q, kv, None, idx, None, scale, causal, d_v)
    g = m.dsa_bwd(q, kv, o, do, lse, None, idx, None, scale, causal, d_v)
    qh = np.ascontiguousarray(q.transpose(1, 0, 2))                  # [H, N, d_qk]
    kh = np.broadcast_to(kv, (H, N, d_qk)).copy()
    vpad = np.zeros((N, d_qk)); vpad[:, :d_v] = kv[:, :d_v]
    vh = np.broadcast_to(vpad, (H, N, d_qk)).copy()
    dopad = np.zeros((H, N, d_qk)); dopad[:, :, :d_v] = do.transpose(1, 0, 2)
    ref = oracle.attn_bwd(qh, kh, vh, dopad, scale, causal)
    checks = [
        (o, ref["o"][:, :, :d_v].transpose(1, 0, 2)),
        (lse, ref["lse"].T),
        (g["dq"], ref["dq"].transpose(1, 0, 2)),
        (g["dkv"], ref["dk"].sum(axis=0) + np.pad(ref["dv"][:, :, :d_v].sum(axis=0), ((0, 0), (0, d_qk - d_v)))),
    ]
    return all(np.max(np.abs(a - b)) <= 1e-10 * max(1.0, np.max(np.abs(b))) for a, b in checks)


def pin_zero_query_closed_form(m, causal):
    """q = 0: every valid score is 0, so L_ih = log(n_i + e^{sink_h}) and
    O_ih = sum of the valid v rows / (n_i + e^{sink_h})."""
    c = _tiny_case(True)
    q = np.zeros_like(c["q"])
    o, lse = m.dsa_fwd(q, c["kv"], c["sink"], c["idx"], c["lens"], 0.9, causal, c["d_v"])
    s_kv = c["kv"].shape[0]
    for i in range(q.shape[0]):
        rows = [int(k) for e, k in enumerate(c["idx"][i])
                if e < c["lens"][i] and 0 <= k < s_kv and (not causal or k <= i)]
        n = len(rows)
        vsum = c["kv"][rows, :c["d_v"]].sum(axis=0) if n else np.zeros(c["d_v"])
        for h in range(q.shape[1]):
            z = n + math.exp(c["sink"][h])
            if abs(lse[i, h] - math.log(z)) > 1e-12:
                return False
            if np.max(np.abs(o[i, h] - vsum / z)) > 1e-12:
                return False
    return True


def pin_list_order_invariance(m, causal):
    """Reordering the entries of each row's list (no length limit; padding stays
    padding wherever it moves) changes nothing."""
    c = _tiny_case(True)
    rng = np.random.default_rng(5)
    perm_idx = np.array([rng.permutation(r) for r in c["idx"]])
    out = []
    for idx in (c["idx"], perm_idx):
        o, lse = m.dsa_fwd(c["q"], c["kv"], c["sink"], idx, None, 0.8, causal, c["d_v"])
        g = m.dsa_bwd(c["q"], c["kv"], o, c["do"], lse, c["sink"], idx, None, 0.8, causal, c["d_v"])
        out.append((o, lse, g["dq"], g["dkv"], g["dsink"]))
    return all(np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(a))) for a, b in zip(*out))


def pin_sink_minus_infinity(m, causal):
    """A sink of -inf is no sink: same O and L, and a zero sink gradient."""
    c = _tiny_case(False)
    c["lens"] = np.array([5, 4, 5, 2, 3], dtype=np.int32)   # no empty row (its L would be -inf)
    neg = np.full(c["q"].shape[1], -np.inf)
    o1, l1 = m.dsa_fwd(c["q"], c["kv"], None, c["idx"], c["lens"], 0.6, causal, c["d_v"])
    o2, l2 = m.dsa_fwd(c["q"], c["kv"], neg, c["idx"], c["lens"], 0.6, causal, c["d_v"])
    g1 = m.dsa_bwd(c["q"], c["kv"], o1, c["do"], l1, None, c["idx"], c["lens"], 0.6, causal, c["d_v"])
    g2 = m.dsa_bwd(c["q"], c["kv"], o2, c["do"], l2, neg, c["idx"], c["lens"], 0.6, causal, c["d_v"])
    return (np.array_equal(o1, o2) and np.array_equal(l1, l2) and np.array_equal(g1["dq"], g2["dq"])
            and np.array_equal(g1["dkv"], g2["dkv"]) and g2["dsink"] is not None
            and np.all(g2["dsink"] == 0.0))


def all_pins(m):
    results = []
    for causal in (False, True):
        results.append(pin_finite_differences(m, causal, True))
        results.append(pin_finite_differences(m, causal, False))
        results.append(pin_dense_reduction(m, causal, 6, 4))
        results.append(pin_dense_reduction(m, causal, 4, 4))
        results.append(pin_zero_query_closed_form(m, causal))
        results.append(pin_list_order_invariance(m, causal))
        results.append(pin_sink_minus_infinity(m, causal))
    return results


# --------------------------------------------------------------------------- tests
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sink", [True, False])
def test_finite_differences(causal, sink):
    assert pin_finite_differences(dsa_mod, causal, sink)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d_qk,d_v", [(6, 4), (4, 4)])
def test_dense_reduction(causal, d_qk, d_v):
    assert pin_dense_reduction(dsa_mod, causal, d_qk, d_v)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_closed_form(causal):
    assert pin_zero_query_closed_form(dsa_mod, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_list_order_invariance(causal):
    assert pin_list_order_invariance(dsa_mod, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_sink_minus_infinity(causal):
    assert pin_sink_minus_infinity(dsa_mod, causal)


MUTATIONS = [
    ("dq without scale", "dq[i] = scale * (dS @ K)", "dq[i] = (dS @ K)"),
    ("dK term without scale", "np.add.at(dkv, sel, scale * (dS.T @ q[i]))", "np.add.at(dkv, sel, (dS.T @ q[i]))"),
    ("dV term dropped", "np.add.at(dkv[:, :d_v], sel, P.T @ do[i])", "pass"),
    ("causal off by one", "ok &= k <= i", "ok &= k < i"),
    ("length off by one", "ok = (e < length)", "ok = (e <= length)"),
    ("sink left out of L", "cols = [S] if snk is None else [S, snk[:, None]]", "cols = [S]"),
    ("dsink sign", "dsink = -np.sum(psink * D, axis=0)", "dsink = np.sum(psink * D, axis=0)"),
    ("V from the last columns", "dP = do[i] @ K[:, :d_v].T", "dP = do[i] @ K[:, -d_v:].T"),
    ("D term dropped", "dS = P * (dP - D[i][:, None])", "dS = P * dP"),
    ("S without scale", "S = scale * (q[i] @ K.T)                       # [H, n]\n        P = np.exp",
     "S = (q[i] @ K.T)\n        P = np.exp"),
]


def _mutant(src, old, new):
    assert src.count(old) >= 1, old
    mod = types.ModuleType("dsa_mutant")
    exec(compile(src.replace(old, new), "dsa_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistakes(name, old, new):
    src = open(SRC).read()
    mod = _mutant(src, old, new)
    with np.errstate(all="ignore"):
        try:
            results = all_pins(mod)
        except Exception:
            results = [False]
    assert not all(results), f"no pin fails with the planted mistake: {name}"
