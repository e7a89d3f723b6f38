"""CUDA path vs the FP64 oracle at the full sizes of the workload list, in the
launch configuration bench.py times (persistent grid over every head).

Per configuration:
  * whole heads: dQ, dK and dV of every row of at least two heads (head 0 and
    the last head; two more seeded heads where N <= 8192) from the oracle's
    row-set entry point, the rows split over threads and the dK / dV
    contributions summed; O and L of every row of head 0 and of the last head;
  * sampled query rows (first and last rows, tile edges, random rows) of those
    heads and two more: O, L and dQ, each needing one row of S, P, dP, dS;
and, on every head, properties that hold at any size: no NaN / unwritten
element, and sum_j dK_j = 0 (rows of dS sum to zero).
The worst error of each quantity over the checked heads is printed.
"""
import math
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from attn_cases import (TOL_GRAD_RELFRO, TOL_L_MAXABS, o_tolerance, rel_fro, to_device, to_f64,
                        whole_head_bwd)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CONFIGS = [
    # id, B, H, N, d, causal, dtype, sigma_qk
    ("causal_b8h16n4096d128", 8, 16, 4096, 128, True, "bf16", 1.0),
    ("noncausal_b4h16n4096d128", 4, 16, 4096, 128, False, "bf16", 1.0),
    ("noncausal_b2h16n8192d128", 2, 16, 8192, 128, False, "bf16", 1.0),
    ("noncausal_b1h16n16384d128", 1, 16, 16384, 128, False, "bf16", 1.0),
    ("fp16_causal_b4h16n1024d64", 4, 16, 1024, 64, True, "fp16", 1.0),
    ("fp16_causal_b4h16n2048d64", 4, 16, 2048, 64, True, "fp16", 1.0),
    ("fp16_causal_b4h16n4096d64", 4, 16, 4096, 64, True, "fp16", 1.0),
    ("stress_b1h32n32768d128", 1, 32, 32768, 128, True, "bf16", 2.0),
    # N not a multiple of 128
    ("ragged_causal_b2h16n4000d128", 2, 16, 4000, 128, True, "bf16", 1.0),
    ("ragged_noncausal_b2h8n3001d64", 2, 8, 3001, 64, False, "fp16", 1.0),
]
SEED = 20261202


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _sample_heads(BH):
    rng = np.random.default_rng(BH)
    extra = [int(x) for x in rng.choice(BH, size=min(2, BH), replace=False)]
    return sorted(set([0, BH - 1] + extra))


def _sample_rows(N, rng):
    rows = {0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1, (N - 1) // 128 * 128}
    rows.update(int(x) for x in rng.integers(0, N, size=22))
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


def _whole_heads(BH, N):
    """Heads checked whole: head 0 and the last head, plus two seeded ones when N <= 8192."""
    heads = {0, BH - 1}
    if N <= 8192:
        rng = np.random.default_rng(7 * BH + N)
        heads.update(int(x) for x in rng.choice(BH, size=min(2, BH), replace=False))
    return sorted(heads)


@pytest.mark.parametrize("cid,B,H,N,d,causal,dtype,sigma", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_full_size_against_oracle(attn, cid, B, H, N, d, causal, dtype, sigma):
    BH = B * H
    scale = 1.0 / math.sqrt(d)
    threads = min(16, os.cpu_count() or 1)
    bits = {n: si.tensor_heads(SEED, n, BH, N, d, sigma if n in ("q", "k") else 1.0, dtype, threads=threads)
            for n in ("q", "k", "v", "do")}
    q, k, v, do = (to_device(bits[n], B, H, dtype) for n in ("q", "k", "v", "do"))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, scale, causal)
    attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0

    # properties on every head
    for name, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(t).all()), f"{name}: unwritten or non-finite elements"
    dkf = dk.float()
    colsum = dkf.sum(dim=2).abs()
    colabs = dkf.abs().sum(dim=2) + 1e-6
    assert float((colsum / colabs).max()) < 2e-2, "sum_j dK_j != 0"

    og, lg = to_f64(o).reshape(BH, N, d), to_f64(lse).reshape(BH, N)
    dqg, dkg, dvg = (to_f64(t).reshape(BH, N, d) for t in (dq, dk, dv))
    del o, lse, dq, dk, dv, ws
    x_of = lambda h: {n: si.bits_to_f32(bits[n][h], dtype).astype(np.float64) for n in bits}
    worst = {n: 0.0 for n in ("o", "l", "dq_rows", "dq", "dk", "dv")}
    per_head = []

    # sampled rows: O, L, dQ
    rng = np.random.default_rng(N + d)
    for h in _sample_heads(BH):
        x = x_of(h)
        rows = _sample_rows(N, rng)
        o_r, l_r, dq_r = oracle.attn_rows(x["q"], x["k"], x["v"], rows, scale, causal, dout=x["do"])
        err = np.abs(og[h][rows] - o_r)
        assert np.all(err <= o_tolerance(o_r, dtype)), (h, float(err.max()))
        worst["o"] = max(worst["o"], float(err.max()))
        le = float(np.max(np.abs(lg[h][rows] - l_r)))
        assert le <= TOL_L_MAXABS, (h, le)
        worst["l"] = max(worst["l"], le)
        e = rel_fro(dqg[h][rows], dq_r)
        assert e <= TOL_GRAD_RELFRO, (h, "dq rows", e)
        worst["dq_rows"] = max(worst["dq_rows"], e)

    # whole heads: dQ, dK, dV of every row; O and L of every row of the first and last head
    for h in _whole_heads(BH, N):
        x = x_of(h)
        if h in (0, BH - 1):
            o_r, l_r, _ = oracle.attn_rows(x["q"], x["k"], x["v"], np.arange(N, dtype=np.int64), scale, causal)
            err = np.abs(og[h] - o_r)
            assert np.all(err <= o_tolerance(o_r, dtype)), (h, "whole-head O", float(err.max()))
            worst["o"] = max(worst["o"], float(err.max()))
            le = float(np.max(np.abs(lg[h] - l_r)))
            assert le <= TOL_L_MAXABS, (h, "whole-head L", le)
            worst["l"] = max(worst["l"], le)
        dq_r, dk_r, dv_r = whole_head_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, threads)
        errs = {}
        for name, got, ref in (("dq", dqg[h], dq_r), ("dk", dkg[h], dk_r), ("dv", dvg[h], dv_r)):
            errs[name] = rel_fro(got, ref)
            worst[name] = max(worst[name], errs[name])
        per_head.append((h, errs))
        for name, e in errs.items():
            assert e <= TOL_GRAD_RELFRO, (h, name, "whole head", e)
    print(f"\n{cid}: worst O max-abs {worst['o']:.4g}, L max-abs {worst['l']:.3g}, dQ rows {worst['dq_rows']:.3g}; "
          f"whole heads rel. Frobenius dQ {worst['dq']:.3g} dK {worst['dk']:.3g} dV {worst['dv']:.3g} "
          f"(heads {[h for h, _ in per_head]})")


def test_largest_supported_size(attn):
    """B H N_pad d just below 2^31 elements, the documented limit: every kernel's 64-bit
    offsets.  131071 heads of N = 128, d = 128 (4.3 GB per tensor).  Every head is checked
    on the device (finite outputs, sum_j dK_j = 0); sampled heads, whose inputs come from the
    seeded generator, against the oracle."""
    B, H, N, d, causal, dtype = 1, 131071, 128, 128, True, "bf16"
    assert B * H * N * d < 2 ** 31
    scale = 1.0 / math.sqrt(d)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(99)
    heads = [0, 1, 65535, H - 2, H - 1]
    x = {n: si.tensor_heads(SEED, n, B * H, N, d, 1.0, dtype, heads=heads) for n in ("q", "k", "v", "do")}
    t = {}
    for n in ("q", "k", "v", "do"):
        t[n] = torch.randn((B, H, N, d), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
        for idx, h in enumerate(heads):
            t[n][0, h] = torch.from_numpy(np.ascontiguousarray(x[n][idx]).view(np.int16)).to("cuda").view(torch.bfloat16)
    o = torch.full_like(t["q"], float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd(t["q"], t["k"], t["v"], o, lse, scale, causal)
    dq, dk, dv = (torch.full_like(t["q"], float("nan")) for _ in range(3))
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    attn.attn_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, ws, scale, causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    del ws
    for name, tt in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(tt).all()), f"{name}: unwritten or non-finite elements"
    colsum = dk.float().sum(dim=2).abs()
    colabs = dk.float().abs().sum(dim=2) + 1e-6
    assert float((colsum / colabs).max()) < 2e-2, "sum_j dK_j != 0"
    for idx, h in enumerate(heads):
        ref = oracle.attn_bwd(*(si.bits_to_f32(x[n][idx], dtype).astype(np.float64) for n in ("q", "k", "v", "do")),
                              scale, causal)
        assert np.max(np.abs(to_f64(o[0, h]) - ref["o"])) <= o_tolerance(ref["o"], dtype).max(), h
        assert np.max(np.abs(to_f64(lse[0, h]) - ref["lse"])) <= TOL_L_MAXABS, h
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert rel_fro(to_f64(got[0, h]), ref[name]) <= TOL_GRAD_RELFRO, (h, name)
