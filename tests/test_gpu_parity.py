"""CUDA path vs the FP64 oracle, element by element, through the C ABI.

Small cases (the oracle runs whole heads in seconds) cover several tiles, a
ragged last Q-tile pair (an odd number of 128-row tiles), causal and
non-causal, d = 64 and 128, bf16 and fp16.  Tolerances: O max-abs 1e-2,
L max-abs 1e-3, dQ/dK/dV relative Frobenius 1e-2 (whole tensor and per head).
Outputs are pre-filled with NaN sentinels so an unwritten element fails.
"""
import math

import numpy as np
import pytest

import oracle
from attn_cases import (TOL_GRAD_RELFRO, TOL_L_MAXABS, TOL_O_MAXABS, f64, input_bits, o_tolerance, rel_fro, to_device,
                        to_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, N, d, causal, dtype
    (1, 2, 128, 64, True, "bf16"),     # the tiny oracle-check workload
    (1, 2, 128, 64, False, "bf16"),
    (1, 2, 384, 128, True, "bf16"),    # 3 tiles: ragged Q-tile pair
    (1, 2, 384, 128, False, "bf16"),
    (2, 3, 512, 128, True, "bf16"),
    (1, 2, 640, 64, True, "fp16"),
    (1, 2, 256, 64, False, "fp16"),
    (1, 1, 1024, 128, True, "bf16"),
    # N not a multiple of 128: ragged last tile (zero-filled loads, masked keys, unstored rows)
    (1, 2, 1, 128, True, "bf16"),
    (1, 2, 1, 64, False, "bf16"),
    (2, 2, 77, 64, True, "bf16"),
    (1, 3, 200, 128, False, "bf16"),
    (1, 2, 333, 128, True, "bf16"),
    (2, 1, 257, 128, True, "fp16"),
    (1, 2, 1000, 64, False, "fp16"),
    # more work units than SMs, so a CTA runs several items and the forward's K/V pairs span
    # item boundaries (a V with the next item's first K): one key tile per item, two, and an
    # odd tile count
    (1, 400, 128, 64, False, "bf16"),
    (1, 200, 256, 128, True, "bf16"),
    (2, 160, 384, 64, True, "fp16"),
]


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _run(attn, B, H, N, d, causal, dtype, seed, sigma_qk=1.0):
    bits = input_bits(seed, B * H, N, d, dtype, sigma_qk=sigma_qk)
    q, k, v, do = (to_device(bits[n], B, H, dtype) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, scale, causal)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    return bits, scale, dict(o=to_f64(o), lse=to_f64(lse), dq=to_f64(dq), dk=to_f64(dk), dv=to_f64(dv))


@pytest.mark.parametrize("B,H,N,d,causal,dtype", SMALL)
def test_fwd_bwd_match_oracle(attn, B, H, N, d, causal, dtype):
    bits, scale, got = _run(attn, B, H, N, d, causal, dtype, seed=1000 + N + d)
    ref = oracle.attn_bwd(*(f64(bits[n], dtype) for n in ("q", "k", "v", "do")), scale, causal)
    shp = (B, H, N, d)
    for name in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[name]).all(), f"{name} has unwritten / non-finite elements"
    o_err = np.max(np.abs(got["o"] - ref["o"].reshape(shp)))
    l_err = np.max(np.abs(got["lse"] - ref["lse"].reshape(B, H, N)))
    assert o_err <= TOL_O_MAXABS, o_err
    assert l_err <= TOL_L_MAXABS, l_err
    for name in ("dq", "dk", "dv"):
        r = ref[name].reshape(shp)
        e = rel_fro(got[name], r)
        assert e <= TOL_GRAD_RELFRO, (name, e)
        for b in range(B):
            for h in range(H):
                eh = rel_fro(got[name][b, h], r[b, h])
                assert eh <= TOL_GRAD_RELFRO, (name, b, h, eh)


def test_sum_of_dk_is_zero(attn):
    """sum_j dK_j = 0 per head (rows of dS sum to zero), on every head."""
    B, H, N, d = 2, 4, 1024, 128
    _, _, got = _run(attn, B, H, N, d, True, "bf16", seed=77)
    s = got["dk"].sum(axis=2)                       # [B, H, d]
    scale_ref = np.abs(got["dk"]).sum(axis=2) + 1e-6
    assert np.max(np.abs(s) / scale_ref) < 2e-2


def test_repeat_is_deterministic_fwd(attn):
    B, H, N, d = 1, 2, 512, 128
    bits = input_bits(5, B * H, N, d)
    q, k, v = (to_device(bits[n], B, H) for n in ("q", "k", "v"))
    o1, l1 = attn.forward(q, k, v, causal=True)
    o2, l2 = attn.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_wide_logits_and_late_spike(attn):
    """Adversarial regimes: sigma = 2 scores, and a key in the last tile aligned
    with some queries so their row max arrives last (forces a rescale)."""
    import seeded_inputs as si
    B, H, N, d, causal = 1, 2, 512, 128, True
    bits = input_bits(31, B * H, N, d, sigma_qk=2.0)
    rows = list(range(N - 128, N, 7))
    for h in range(B * H):
        bits["k"][h] = si.late_spike(bits["q"][h], bits["k"][h], "bf16", 30.0, rows)
    q, k, v, do = (to_device(bits[n], B, H) for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o, lse = attn.forward(q, k, v, scale, causal)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, scale, causal)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(*(f64(bits[n]) for n in ("q", "k", "v", "do")), scale, causal)
    shp = (B, H, N, d)
    o_ref = ref["o"].reshape(shp)
    o_err = np.abs(to_f64(o) - o_ref)
    print("late spike: O max-abs", o_err.max(), "max |O_ref|", np.abs(o_ref).max())
    assert np.all(o_err <= o_tolerance(o_ref)), o_err.max()
    assert np.max(np.abs(to_f64(lse) - ref["lse"].reshape(B, H, N))) <= TOL_L_MAXABS
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        e = rel_fro(to_f64(t), ref[name].reshape(shp))
        print("late spike:", name, e)
        assert e <= TOL_GRAD_RELFRO, name
