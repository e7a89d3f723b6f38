"""The BSHD and packed variable-length layouts at full size, against the FP64 oracle and the
[B, H, N, d] path, through the C ABI.

Workloads, as the sweep times them (causal, bf16, H = 16, d = 128):
  * BSHD [B, N, H, d] with B = 8, N = 4096 (the bench workload in the token-major layout);
  * 32 packed sequences of 512, 752, ..., 7952 tokens (135424 rows, most sequences ending in a
    ragged tile), whose units the kernels take from the launch's work counter.
Per workload:
  * every element written (NaN pre-fill) and finite;
  * against the [B, H, N, d] path on the same slices: O, L, dK and dV bit for bit, and dQ within
    DQ_CROSS.  Only the row addressing (and, for packed sequences, the work distribution) differs,
    and the arithmetic order of everything but dQ's FP32 reductions is fixed;
  * whole slices against the oracle: O and L of every row, and dQ, dK, dV of every row, of two
    (sequence, head) slices.
Inputs come from the seeded generator, one (sequence, head) slice at a time.
"""
import math
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from attn_cases import TOL_GRAD_RELFRO, TOL_L_MAXABS, o_tolerance, rel_fro, to_f64, whole_head_bwd

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SEED = 31
DQ_CROSS = 2e-3
H, D = 16, 128
PACKED_LENS = [512 + 240 * i for i in range(32)]


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _dev16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def _fwd_bwd(attn, t, lse_shape, layout, cu=None, maxlen=None, B=None, N=None):
    """Forward and backward on device tensors t[name]; layout "bhsd" uses attn_fwd / attn_bwd."""
    scale = 1.0 / math.sqrt(D)
    o = torch.full_like(t["q"], float("nan"))
    lse = torch.full(lse_shape, float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.full_like(t["q"], float("nan")) for _ in range(3))
    if layout == "bhsd":
        ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, D), dtype=torch.uint8, device="cuda")
        attn.attn_fwd(t["q"], t["k"], t["v"], o, lse, scale, True)
        attn.attn_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, ws, scale, True)
    else:
        total = t["q"].shape[0] if layout == "packed" else B * N
        ws = torch.empty(attn.attn_bwd_layout_workspace_size(B, H, maxlen, D, layout, total), dtype=torch.uint8,
                         device="cuda")
        attn.attn_fwd_layout(t["q"], t["k"], t["v"], o, lse, scale, True, layout, cu, maxlen)
        attn.attn_bwd_layout(t["q"], t["k"], t["v"], o, t["do"], lse, dq, dk, dv, ws, scale, True, layout, cu,
                             maxlen)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    out = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    for name, x in out.items():
        assert bool(torch.isfinite(x).all()), f"{layout} {name}: unwritten or non-finite elements"
    return out


def _dq_cross(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def _check_slice_against_oracle(x, got, what):
    """x: bits of one (sequence, head) slice, name -> [n, d]; got: that slice's outputs as
    float64 arrays (o, dq, dk, dv: [n, d]; lse: [n])."""
    scale = 1.0 / math.sqrt(D)
    f = {n: si.bits_to_f32(x[n], "bf16").astype(np.float64) for n in x}
    n = f["q"].shape[0]
    o_r, l_r, _ = oracle.attn_rows(f["q"], f["k"], f["v"], np.arange(n, dtype=np.int64), scale, True)
    err = np.abs(got["o"] - o_r)
    assert np.all(err <= o_tolerance(o_r, "bf16")), (what, "O", float(err.max()))
    le = float(np.max(np.abs(got["lse"] - l_r)))
    assert le <= TOL_L_MAXABS, (what, "L", le)
    dq_r, dk_r, dv_r = whole_head_bwd(f["q"], f["k"], f["v"], f["do"], scale, True, min(16, os.cpu_count() or 1))
    errs = {name: rel_fro(got[name], ref) for name, ref in (("dq", dq_r), ("dk", dk_r), ("dv", dv_r))}
    for name, e in errs.items():
        assert e <= TOL_GRAD_RELFRO, (what, name, e)
    return float(err.max()), le, errs


def test_bshd_full_size(attn):
    B, N = 8, 4096
    bits = {n: si.tensor_heads(SEED, n, B * H, N, D, 1.0, "bf16", threads=min(16, os.cpu_count() or 1))
            for n in ("q", "k", "v", "do")}
    bhsd = {n: _dev16(bits[n]).reshape(B, H, N, D) for n in bits}
    ref = _fwd_bwd(attn, bhsd, (B, H, N), "bhsd", B=B, N=N)
    bshd = {n: t.transpose(1, 2).contiguous() for n, t in bhsd.items()}
    del bhsd
    got = _fwd_bwd(attn, bshd, (B, H, N), "bshd", maxlen=N, B=B, N=N)
    del bshd
    for name in ("o", "dk", "dv"):
        assert torch.equal(got[name].transpose(1, 2), ref[name]), f"{name} differs from the [B, H, N, d] path"
    assert torch.equal(got["lse"], ref["lse"])
    e = _dq_cross(got["dq"].transpose(1, 2), ref["dq"])
    assert e <= DQ_CROSS, e
    for bh in (0, B * H - 1):
        b, h = divmod(bh, H)
        sl = {name: to_f64(got[name][b, :, h]) for name in ("o", "dq", "dk", "dv")}
        sl["lse"] = to_f64(got["lse"][b, h])
        o_err, l_err, errs = _check_slice_against_oracle({n: bits[n][bh] for n in bits}, sl, f"head {bh}")
        print(f"\nBSHD head {bh}: O {o_err:.3g}, L {l_err:.3g}, dQ {errs['dq']:.3g} dK {errs['dk']:.3g} "
              f"dV {errs['dv']:.3g}; dQ vs [B, H, N, d] {e:.3g}")


def test_packed_full_size(attn):
    lens = PACKED_LENS
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    total, maxlen, B = int(cu[-1]), max(lens), len(lens)
    slices = [{n: si.tensor_heads(SEED + 1 + b, n, H, lens[b], D, 1.0, "bf16") for n in ("q", "k", "v", "do")}
              for b in range(B)]
    packed = {}
    for name in ("q", "k", "v", "do"):
        arr = np.empty((total, H, D), dtype=np.uint16)
        for b in range(B):
            arr[cu[b]:cu[b + 1]] = slices[b][name].transpose(1, 0, 2)   # [H, n, d] -> [n, H, d]
        packed[name] = _dev16(arr)
    cu_dev = torch.from_numpy(cu.astype(np.int32)).to("cuda")
    got = _fwd_bwd(attn, packed, (H, total), "packed", cu=cu_dev, maxlen=maxlen, B=B)
    del packed
    worst_dq = 0.0
    for b, n in enumerate(lens):
        t = {name: _dev16(slices[b][name]).reshape(1, H, n, D) for name in slices[b]}
        ref = _fwd_bwd(attn, t, (1, H, n), "bhsd", B=1, N=n)
        rows = slice(int(cu[b]), int(cu[b + 1]))
        for name in ("o", "dk", "dv"):
            mine = got[name][rows].transpose(0, 1)                           # [H, n, d]
            assert torch.equal(mine, ref[name][0]), (b, name)
        assert torch.equal(got["lse"][:, rows], ref["lse"][0]), (b, "lse")
        e = _dq_cross(got["dq"][rows].transpose(0, 1), ref["dq"][0])
        assert e <= DQ_CROSS, (b, "dq", e)
        worst_dq = max(worst_dq, e)
    # whole slices against the oracle: the longest sequence's head 0 and a ragged one's last head
    for b, h in ((B - 1, 0), (1, H - 1)):
        rows = slice(int(cu[b]), int(cu[b + 1]))
        sl = {name: to_f64(got[name][rows, h]) for name in ("o", "dq", "dk", "dv")}
        sl["lse"] = to_f64(got["lse"][h, rows])
        o_err, l_err, errs = _check_slice_against_oracle({n: slices[b][n][h] for n in slices[b]}, sl,
                                                         f"sequence {b} head {h}")
        print(f"\npacked sequence {b} ({lens[b]} tokens) head {h}: O {o_err:.3g}, L {l_err:.3g}, "
              f"dQ {errs['dq']:.3g} dK {errs['dk']:.3g} dV {errs['dv']:.3g}; worst dQ vs [B, H, N, d] {worst_dq:.3g}")
