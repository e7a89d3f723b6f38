"""Shared test helpers: seeded inputs for both sides, oracle calls, error norms.

Imports the oracle (test infrastructure) and the seeded input generator; the
CUDA side is reached only through the package binding.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle
import seeded_inputs as si


def input_bits(seed, BH, N, d, dtype="bf16", sigma_qk=1.0, sigma_vdo=1.0, heads=None):
    """16-bit patterns of q, k, v, dO: dict name -> [n_heads, N, d] uint16."""
    out = {}
    for name, sig in (("q", sigma_qk), ("k", sigma_qk), ("v", sigma_vdo), ("do", sigma_vdo)):
        out[name] = si.tensor_heads(seed, name, BH, N, d, sig, dtype, heads=heads)
    return out


def f64(bits, dtype="bf16"):
    return si.bits_to_f32(bits, dtype).astype(np.float64)


def to_device(bits, B, H, dtype="bf16"):
    import torch
    N, d = bits.shape[-2], bits.shape[-1]
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).reshape(B, H, N, d)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return t.to("cuda").view(tdt)


def to_f64(t):
    """A CUDA 16-bit / fp32 tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def rel_fro(x, ref):
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den > 0 else 1.0))


# Tolerances (fixed by the benchmark spec of the method for unit-normal inputs)
TOL_O_MAXABS = 1e-2
TOL_L_MAXABS = 1e-3
TOL_GRAD_RELFRO = 1e-2


def o_tolerance(o_ref, dtype="bf16"):
    """Element-wise bound on |O_gpu - O_ref|: the stated 1e-2 for unit-normal
    inputs, plus the rounding of the 16-bit output itself (unit roundoff 2^-8 |O|
    for bf16, 2^-11 |O| for fp16), which no kernel can avoid once |O| grows past
    2 (as it does for the sigma = 2 inputs)."""
    half_ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    return TOL_O_MAXABS + half_ulp * np.abs(o_ref)


def whole_head_bwd(q, k, v, do, scale, causal, threads):
    """dQ, dK, dV of every row of one head from the oracle's row-set entry point.  Rows are
    dealt round robin to the threads (so causal rows of different cost spread evenly); each
    thread returns its rows' dQ and their contributions to dK and dV, which are summed."""
    N = q.shape[0]
    chunks = [np.arange(t, N, threads, dtype=np.int64) for t in range(min(threads, N))]

    def one(rows):
        return oracle.attn_bwd_rowset(q, k, v, do, rows, scale, causal)

    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(one, chunks))
    dq = np.empty_like(q)
    for rows, p in zip(chunks, parts):
        dq[rows] = p[0]
    return dq, sum(p[1] for p in parts), sum(p[2] for p in parts)
