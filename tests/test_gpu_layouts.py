"""The BSHD and packed variable-length layouts vs the FP64 oracle, through the C ABI.

Inputs come from the same seeded generator as the [B, H, N, d] tests, one
(sequence, head) slice at a time, arranged in the layout under test; the oracle
runs every slice on its own.  Tolerances as in test_gpu_parity.  Each layout is
also checked against the [B, H, N, d] path on the same slices: only the row
addressing differs, so O, L, dK and dV agree bit for bit.  dQ adds FP32 partials
in no fixed order, so after rounding to 16 bits single elements may differ by one
unit in the last place (2^-8 relative for bf16); the two paths' dQ are compared
with a relative Frobenius bound of DQ_CROSS = 2e-3 (the oracle bound is 1e-2).  Outputs are
pre-filled with NaN so an unwritten element fails.
"""
import math

import numpy as np
import pytest

import oracle
from attn_cases import TOL_GRAD_RELFRO, TOL_L_MAXABS, TOL_O_MAXABS, f64, input_bits, rel_fro, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BSHD_CASES = [
    # B, H, N, d, causal, dtype
    (2, 3, 333, 128, True, "bf16"),
    (1, 2, 512, 128, False, "bf16"),
    (2, 2, 77, 64, True, "bf16"),
    (1, 2, 256, 64, False, "fp16"),
    (2, 100, 200, 64, True, "bf16"),  # 200 units: several items per CTA, ragged tiles
]
DQ_CROSS = 2e-3
PACKED_CASES = [
    # sequence lengths, H, d, causal, dtype, max_seqlen slack
    ([1, 128, 300, 0, 257], 2, 128, True, "bf16", 0),
    ([500, 3, 129], 3, 64, False, "fp16", 100),
    ([640, 384], 1, 128, True, "bf16", 0),
    ([0, 0, 5], 2, 64, True, "bf16", 0),
    ([200, 1000, 77, 128], 2, 128, False, "bf16", 24),
]


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _dev(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda")
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def _nan_like(t):
    return torch.full_like(t, float("nan"))


def _bhsd_run(attn, x, B, H, N, d, scale, causal, dtype):
    """The [B, H, N, d] path on bits x[name] of shape [B H, N, d]: dict of float64 arrays."""
    q, k, v, do = (_dev(x[n].reshape(B, H, N, d), dtype) for n in ("q", "k", "v", "do"))
    o, lse = _nan_like(q), torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o, lse, scale, causal)
    dq, dk, dv = _nan_like(q), _nan_like(q), _nan_like(q)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    return dict(o=to_f64(o), lse=to_f64(lse), dq=to_f64(dq), dk=to_f64(dk), dv=to_f64(dv))


def _check_grads(got, ref, what):
    for name in ("dq", "dk", "dv"):
        e = rel_fro(got[name], ref[name])
        assert e <= TOL_GRAD_RELFRO, (what, name, e)


@pytest.mark.parametrize("B,H,N,d,causal,dtype", BSHD_CASES)
def test_bshd_matches_oracle_and_bhsd(attn, B, H, N, d, causal, dtype):
    scale = 1.0 / math.sqrt(d)
    x = input_bits(4000 + N + d, B * H, N, d, dtype)
    # [B H, N, d] -> [B, N, H, d]
    q, k, v, do = (_dev(x[n].reshape(B, H, N, d).transpose(0, 2, 1, 3), dtype) for n in ("q", "k", "v", "do"))
    o, lse = _nan_like(q), torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_layout(q, k, v, o, lse, scale, causal, "bshd")
    dq, dk, dv = _nan_like(q), _nan_like(q), _nan_like(q)
    ws = torch.empty(attn.attn_bwd_layout_workspace_size(B, H, N, d, "bshd", B * N), dtype=torch.uint8,
                     device="cuda")
    attn.attn_bwd_layout(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, "bshd")
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    # back to [B, H, N, d]
    got = {n: to_f64(t).transpose(0, 2, 1, 3) for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    got["lse"] = to_f64(lse)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert np.isfinite(got[n]).all(), f"{n}: unwritten or non-finite elements"

    ref = oracle.attn_bwd(*(f64(x[n], dtype) for n in ("q", "k", "v", "do")), scale, causal)
    shp = (B, H, N, d)
    assert np.max(np.abs(got["o"] - ref["o"].reshape(shp))) <= TOL_O_MAXABS
    assert np.max(np.abs(got["lse"] - ref["lse"].reshape(B, H, N))) <= TOL_L_MAXABS
    _check_grads(got, {n: ref[n].reshape(shp) for n in ("dq", "dk", "dv")}, "oracle")

    base = _bhsd_run(attn, x, B, H, N, d, scale, causal, dtype)
    for n in ("o", "lse", "dk", "dv"):
        assert np.array_equal(got[n], base[n]), f"{n} differs from the [B, H, N, d] path"
    assert rel_fro(got["dq"], base["dq"]) <= DQ_CROSS


@pytest.mark.parametrize("lens,H,d,causal,dtype,slack", PACKED_CASES)
def test_packed_matches_oracle_and_bhsd(attn, lens, H, d, causal, dtype, slack):
    scale = 1.0 / math.sqrt(d)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    B = len(lens)
    max_seqlen = max(max(lens), 1) + slack
    slices = [input_bits(5000 + 7 * b + n, H, n, d, dtype) if n > 0 else None for b, n in enumerate(lens)]
    packed = {}
    for name in ("q", "k", "v", "do"):
        arr = np.zeros((total, H, d), dtype=np.uint16)
        for b, n in enumerate(lens):
            if n:
                arr[cu[b]:cu[b + 1]] = slices[b][name].transpose(1, 0, 2)   # [H, n, d] -> [n, H, d]
        packed[name] = arr
    q, k, v, do = (_dev(packed[n], dtype) for n in ("q", "k", "v", "do"))
    cu_dev = torch.from_numpy(cu).to("cuda")
    o, lse = _nan_like(q), torch.full((H, total), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_layout(q, k, v, o, lse, scale, causal, "packed", cu_dev, max_seqlen)
    dq, dk, dv = _nan_like(q), _nan_like(q), _nan_like(q)
    ws = torch.empty(attn.attn_bwd_layout_workspace_size(B, H, max_seqlen, d, "packed", total), dtype=torch.uint8,
                     device="cuda")
    attn.attn_bwd_layout(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, "packed", cu_dev, max_seqlen)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    got = {n: to_f64(t) for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    got_lse = to_f64(lse)
    for n in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[n]).all(), f"{n}: unwritten or non-finite elements"
    assert np.isfinite(got_lse).all()

    for b, n in enumerate(lens):
        if n == 0:
            continue
        rows = slice(cu[b], cu[b + 1])
        mine = {name: got[name][rows].transpose(1, 0, 2) for name in ("o", "dq", "dk", "dv")}  # [H, n, d]
        mine["lse"] = got_lse[:, rows]
        x = slices[b]
        ref = oracle.attn_bwd(*(f64(x[nm], dtype) for nm in ("q", "k", "v", "do")), scale, causal)
        assert np.max(np.abs(mine["o"] - ref["o"])) <= TOL_O_MAXABS, b
        assert np.max(np.abs(mine["lse"] - ref["lse"])) <= TOL_L_MAXABS, b
        _check_grads(mine, ref, f"sequence {b}")
        base = _bhsd_run(attn, x, 1, H, n, d, scale, causal, dtype)
        for name in ("o", "lse", "dk", "dv"):
            assert np.array_equal(mine[name], base[name].reshape(mine[name].shape)), (b, name)
        assert rel_fro(mine["dq"], base["dq"].reshape(mine["dq"].shape)) <= DQ_CROSS


def test_packed_bad_offsets_are_reported_and_skipped(attn):
    """Offsets that decrease, or a sequence longer than max_seqlen: those sequences are
    skipped (no load or store touches them) and the device error word says so; the
    valid sequence is still computed."""
    H, d, dtype = 2, 64, "bf16"
    cu = np.array([0, 100, 50, 200], dtype=np.int32)   # seq 1 decreasing, seq 2 150 rows > max 128
    total, max_seqlen, scale = 200, 128, 1.0 / math.sqrt(d)
    x = input_bits(6000, H, 100, d, dtype)
    packed = {}
    for name in ("q", "k", "v"):
        arr = np.zeros((total, H, d), dtype=np.uint16)
        arr[:100] = x[name].transpose(1, 0, 2)
        packed[name] = _dev(arr, dtype)
    o = _nan_like(packed["q"])
    lse = torch.full((H, total), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_layout(packed["q"], packed["k"], packed["v"], o, lse, scale, True, "packed",
                         torch.from_numpy(cu).to("cuda"), max_seqlen)
    assert attn.attn_last_device_error() == 1          # ATTN_ERR_INVALID_ARG
    assert attn.attn_last_device_error() == 0          # the word is cleared by the read
    got = to_f64(o)
    assert np.isfinite(got[:100]).all()
    assert np.isnan(got[100:]).all()                   # rows of the skipped sequences untouched
    ref_o, ref_l = oracle.attn_fwd(*(f64(x[n], dtype) for n in ("q", "k", "v")), scale, True)
    assert np.max(np.abs(got[:100].transpose(1, 0, 2) - ref_o)) <= TOL_O_MAXABS
