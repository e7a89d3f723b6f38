"""FP64 CPU oracle for sparse top-k attention with a shared latent key/value row
(forward and backward).

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import it; the product path never does, and nothing here
imports the product path.

What it computes follows the workload of "Improve performance of SM100 DSA
backward kernel" (cudnn-frontend pull request 684, PR description: gathered
keys by top-k index, attention sink, QK width 512 or 576 with V = the first 512
columns, per-row top-k lengths, causal or not, dQ / dKV / dSink outputs), with
the attention equations of "Writing Speed-of-Light Attention Backward Kernel for
5090 in CUDA" (section "Mathematical Formulation") applied to the gathered keys.
For query row i and head h, over the valid entries e of row i's index list
(position e < len_i, 0 <= idx[i, e] < s_kv, and idx[i, e] <= i when causal),
with k_e = kv[idx[i, e]] and v_e = k_e[:d_v]:

    S_e   = scale * q_ih . k_e
    L_ih  = log( sum_e exp(S_e) + exp(sink_h) )        (no sink term without sinks)
    P_e   = exp(S_e - L_ih),   O_ih = sum_e P_e v_e

and, given O and L (the backward's inputs, as in the dense method):

    D_ih   = dO_ih . O_ih
    dP_e   = dO_ih . v_e,      dS_e = P_e (dP_e - D_ih)
    dq_ih  = scale * sum_e dS_e k_e
    dkv[idx[i, e]] += scale * dS_e q_ih  (all d_qk columns) + P_e dO_ih (first d_v columns)
    dsink_h = - sum_i exp(sink_h - L_ih) D_ih

The sink is a logit with no value row: its dP is 0, so its dS is -P_sink D.
Every entry of the list counts, so a key listed twice is attended twice.

Parity pins: ``tests/test_oracle_dsa.py`` (finite differences of a scalar loss
through ``dsa_fwd``, reduction to the dense oracle when every row lists all
keys in order, the q = 0 closed form with a sink, invariance under reordering a
row's list, and sink -> -inf equal to no sink).
"""
from __future__ import annotations

import numpy as np


def _valid(idx_row, length, s_kv, i, causal):
    """Positions e of row i's list that take part (see the module docstring)."""
    e = np.arange(idx_row.shape[0])
    k = idx_row.astype(np.int64)
    ok = (e < length) & (k >= 0) & (k < s_kv)
    if causal:
        ok &= k <= i
    return np.nonzero(ok)[0]


def _row_len(topk_len, i, topk):
    if topk_len is None:
        return topk
    return max(0, min(int(topk_len[i]), topk))


def dsa_fwd(q, kv, sink, idx, topk_len, scale: float, causal: bool, d_v: int):
    """q [s_q, H, d_qk], kv [s_kv, d_qk], sink [H] or None, idx int [s_q, topk],
    topk_len int [s_q] or None.  Returns (O [s_q, H, d_v], L [s_q, H]) in float64."""
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    s_q, H, _ = q.shape
    s_kv = kv.shape[0]
    topk = idx.shape[1]
    snk = None if sink is None else np.asarray(sink, dtype=np.float64)
    O = np.zeros((s_q, H, d_v))
    L = np.empty((s_q, H))
    for i in range(s_q):
        sel = idx[i, _valid(idx[i], _row_len(topk_len, i, topk), s_kv, i, causal)].astype(np.int64)
        K = kv[sel]                                    # [n, d_qk]
        S = scale * (q[i] @ K.T)                       # [H, n]
        cols = [S] if snk is None else [S, snk[:, None]]
        allS = np.concatenate(cols, axis=1)
        if allS.shape[1] == 0:
            L[i] = -np.inf                             # nothing to attend to
            continue
        m = np.max(allS, axis=1, keepdims=True)
        L[i] = (m + np.log(np.sum(np.exp(allS - m), axis=1, keepdims=True)))[:, 0]
        P = np.exp(S - L[i][:, None])
        O[i] = P @ K[:, :d_v]
    return O, L


def dsa_bwd(q, kv, o, do, lse, sink, idx, topk_len, scale: float, causal: bool, d_v: int):
    """Backward given the forward's O and L.  Shapes as in dsa_fwd plus
    o, do [s_q, H, d_v], lse [s_q, H].  Returns dict(dq [s_q, H, d_qk],
    dkv [s_kv, d_qk], dsink [H] or None) in float64."""
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    s_q, H, d_qk = q.shape
    s_kv = kv.shape[0]
    topk = idx.shape[1]
    dq = np.zeros_like(q)
    dkv = np.zeros((s_kv, d_qk))
    D = np.sum(do * o, axis=2)                          # [s_q, H]
    dsink = None
    if sink is not None:
        snk = np.asarray(sink, dtype=np.float64)
        with np.errstate(over="ignore", invalid="ignore"):
            psink = np.where(np.isfinite(lse), np.exp(snk[None, :] - lse), 0.0)
        dsink = -np.sum(psink * D, axis=0)
    for i in range(s_q):
        sel = idx[i, _valid(idx[i], _row_len(topk_len, i, topk), s_kv, i, causal)].astype(np.int64)
        if sel.shape[0] == 0:
            continue
        K = kv[sel]                                    # [n, d_qk]
        S = scale * (q[i] @ K.T)                       # [H, n]
        P = np.exp(S - lse[i][:, None])
        dP = do[i] @ K[:, :d_v].T                      # [H, n]
        dS = P * (dP - D[i][:, None])
        dq[i] = scale * (dS @ K)
        np.add.at(dkv, sel, scale * (dS.T @ q[i]))
        np.add.at(dkv[:, :d_v], sel, P.T @ do[i])
    return dict(dq=dq, dkv=dkv, dsink=dsink)
