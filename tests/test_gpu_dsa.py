"""Sparse top-k attention backward (shared latent key/value rows) vs the FP64 oracle,
through the C ABI.

Inputs: q, kv, dO from the seeded generator (bf16), top-k lists of distinct random
keys (causal rows draw from keys 0..i and are padded with -1), a sink per head.  O and
L are the oracle forward's, rounded as the kernel receives them (O to bf16, L to
FP32), and the oracle backward is given the same rounded values, so both sides
compute the backward of the same inputs.  Some cases add padding entries, indices
outside [0, s_kv), duplicates, keys after the query (masked when causal), shortened
rows and an empty row.  Bounds: dQ and dKV relative Frobenius error <= 1e-2 (the
gradient tolerance of the dense path), dSink <= 1e-3.  Outputs are pre-filled with
NaN so an unwritten element fails.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from attn_cases import TOL_GRAD_RELFRO, rel_fro

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # s_q, s_kv, H, d_qk, topk, causal, sink, perturb
    (40, 300, 64, 576, 256, False, True, False),
    (48, 200, 128, 512, 192, True, True, False),
    (32, 500, 64, 576, 384, False, True, True),
    (24, 64, 64, 512, 128, True, False, True),
    (16, 1000, 128, 576, 100, False, True, True),
]
TOL_DSINK = 1e-3


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(torch.bfloat16)


def _f64(bits):
    return si.bf16_bits_to_f32(bits).astype(np.float64)


def _perturb(idx, lens, s_q, s_kv, seed):
    """Padding, out-of-range indices, duplicates, keys after the query, a shortened
    row and an empty row."""
    rng = np.random.default_rng(seed)
    idx = idx.copy()
    lens = lens.copy()
    topk = idx.shape[1]
    for i in range(s_q):
        e = rng.integers(0, topk, size=4)
        idx[i, e[0]] = -1
        idx[i, e[1]] = s_kv + int(rng.integers(0, 7))
        idx[i, e[2]] = idx[i, e[3]]                        # duplicate (may be -1)
        idx[i, int(rng.integers(0, topk))] = int(rng.integers(0, s_kv))   # possibly after the query
    lens[1] = topk // 3
    lens[2] = 0
    lens[3] = topk + 5                                       # clamped to topk
    return idx, lens


def _run_case(attn, s_q, s_kv, H, d_qk, topk, causal, sink, perturb, seed):
    d_v, scale = 512, 1.0 / math.sqrt(d_qk)
    x = si.dsa_inputs(seed, s_q, s_kv, H, d_qk, d_v, topk, causal)
    idx, lens = x["idx"], x["lens"]
    if perturb:
        idx, lens = _perturb(idx, lens, s_q, s_kv, seed)
    use_len = perturb or causal
    snk = x["sink"].astype(np.float64) if sink else None
    q, kv, do = _f64(x["q"]), _f64(x["kv"]), _f64(x["do"])
    o_ref, l_ref = oracle.dsa_fwd(q, kv, snk, idx, lens if use_len else None, scale, causal, d_v)
    o_bits = si.round_bf16_bits(o_ref.astype(np.float32))
    l32 = l_ref.astype(np.float32)
    ref = oracle.dsa_bwd(q, kv, _f64(o_bits), do, l32.astype(np.float64), snk, idx,
                         lens if use_len else None, scale, causal, d_v)

    dev = dict(q=_bf16_dev(x["q"]), kv=_bf16_dev(x["kv"]), do=_bf16_dev(x["do"]), o=_bf16_dev(o_bits))
    lse = torch.from_numpy(l32).to("cuda")
    sink_t = torch.from_numpy(x["sink"]).to("cuda") if sink else None
    idx_t = torch.from_numpy(np.ascontiguousarray(idx)).to("cuda")
    len_t = torch.from_numpy(np.ascontiguousarray(lens)).to("cuda") if use_len else None
    dq = torch.full((s_q, H, d_qk), float("nan"), dtype=torch.bfloat16, device="cuda")
    dkv = torch.full((s_kv, d_qk), float("nan"), dtype=torch.bfloat16, device="cuda")
    dsink = torch.full((H,), float("nan"), dtype=torch.float32, device="cuda") if sink else None
    ws = torch.empty(attn.attn_dsa_bwd_workspace_size(s_kv, d_qk), dtype=torch.uint8, device="cuda")
    attn.attn_dsa_bwd(dev["q"], dev["kv"], dev["o"], dev["do"], lse, sink_t, idx_t, len_t, dq, dkv, dsink, ws,
                      scale, causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    got_dq = dq.float().cpu().numpy().astype(np.float64)
    got_dkv = dkv.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got_dq).all() and np.isfinite(got_dkv).all()
    e_dq, e_dkv = rel_fro(got_dq, ref["dq"]), rel_fro(got_dkv, ref["dkv"])
    assert e_dq <= TOL_GRAD_RELFRO, ("dq", e_dq)
    assert e_dkv <= TOL_GRAD_RELFRO, ("dkv", e_dkv)
    if perturb:
        assert np.all(got_dq[2] == 0.0)                      # the empty row
    if sink:
        got_ds = dsink.cpu().numpy().astype(np.float64)
        e_ds = rel_fro(got_ds, ref["dsink"])
        assert e_ds <= TOL_DSINK, ("dsink", e_ds)
    return e_dq, e_dkv


@pytest.mark.parametrize("s_q,s_kv,H,d_qk,topk,causal,sink,perturb", CASES)
def test_dsa_bwd_matches_oracle(attn, s_q, s_kv, H, d_qk, topk, causal, sink, perturb):
    _run_case(attn, s_q, s_kv, H, d_qk, topk, causal, sink, perturb, seed=700 + s_q + topk)


def test_dsa_bwd_argument_errors(attn):
    """Unsupported shapes are refused before any launch."""
    q = torch.zeros((4, 32, 576), dtype=torch.bfloat16, device="cuda")   # H = 32: not a multiple of 64
    kv = torch.zeros((8, 576), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((4, 32, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((4, 32), dtype=torch.float32, device="cuda")
    idx = torch.zeros((4, 8), dtype=torch.int32, device="cuda")
    ws = torch.empty(attn.attn_dsa_bwd_workspace_size(8, 576), dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_dsa_bwd(q, kv, o, o, lse, None, idx, None, torch.empty_like(q), torch.empty_like(kv), None, ws,
                          0.1, False)
    assert attn.attn_last_launch_count() == 0


def _sub_bwd(x, rows, idx_rows, scale, causal):
    """The oracle backward of `rows` only (their own lists), inputs taken from the device."""
    t = lambda a: a.float().cpu().numpy().astype(np.float64)
    sel = torch.as_tensor(rows, device="cuda")
    return oracle.dsa_bwd(t(x["q"][sel]), t(x["kv"]), t(x["o"][sel]), t(x["do"][sel]), t(x["lse"][sel]),
                          t(x["sink"]), idx_rows, None, scale, causal, 512)


def _forward_inputs(x, scale, d_v=512, causal=False):
    """The backward's O (bf16) and L (FP32) inputs at full size, from a plain PyTorch FP32
    forward over each row's gathered keys with the sink in the denominator (input
    preparation: the oracle's backward is given these same O and L).  causal: entries naming
    a key after the row's own position take no part."""
    q, kv, sink, idx = x["q"], x["kv"], x["sink"], x["idx"]
    s_q, H = q.shape[0], q.shape[1]
    o = torch.empty((s_q, H, d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((s_q, H), dtype=torch.float32, device="cuda")
    kvf = kv.float()
    for r0 in range(0, s_q, 64):
        r1 = min(s_q, r0 + 64)
        ix = idx[r0:r1].long()
        K = kvf[ix.clamp(min=0)]
        S = torch.einsum("rhd,rkd->rhk", q[r0:r1].float(), K) * scale
        valid = ix >= 0
        if causal:
            valid &= ix <= torch.arange(r0, r1, device="cuda")[:, None]
        S = S.masked_fill(~valid[:, None, :], float("-inf"))
        L = torch.logsumexp(torch.cat([S, sink[None, :, None].expand(r1 - r0, H, 1)], dim=2), dim=2)
        o[r0:r1] = torch.einsum("rhk,rkd->rhd", torch.exp(S - L[:, :, None]), K[:, :, :d_v]).to(torch.bfloat16)
        lse[r0:r1] = L
    return o, lse


def test_dsa_bwd_full_size_sampled(attn):
    """s_q = s_kv = 4096, H = 128, QK 576, top-k 2048 (the largest shape of the pull
    request's table), sink on, launched as bench.py times it.  dQ on sampled queries;
    dKV on sampled keys (L is an input, so each listed (query, key) entry contributes on
    its own: the oracle runs on the queries that list the key, each with that one entry);
    dSink over all rows, 256 at a time."""
    s, H, d_qk, topk = 4096, 128, 576, 2048
    x = si.dsa_device_draws(s, s, H, d_qk, topk, False, seed=17)
    scale = d_qk ** -0.5
    x["o"], x["lse"] = _forward_inputs(x, scale)
    dq = torch.full_like(x["q"], float("nan"))
    dkv = torch.full_like(x["kv"], float("nan"))
    dsink = torch.full_like(x["sink"], float("nan"))
    ws = torch.empty(attn.attn_dsa_bwd_workspace_size(s, d_qk), dtype=torch.uint8, device="cuda")
    attn.attn_dsa_bwd(x["q"], x["kv"], x["o"], x["do"], x["lse"], x["sink"], x["idx"], x["lens"], dq, dkv, dsink, ws,
                      scale, False)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dkv.float()).all()
    idx = x["idx"].cpu().numpy()
    rng = np.random.default_rng(3)

    rows = [0, 1, 2047, s - 1] + [int(r) for r in rng.integers(0, s, 4)]
    ref = _sub_bwd(x, rows, idx[rows], scale, False)
    got = dq[torch.as_tensor(rows, device="cuda")].float().cpu().numpy().astype(np.float64)
    for n, r in enumerate(rows):
        assert rel_fro(got[n], ref["dq"][n]) <= TOL_GRAD_RELFRO, ("dq", r)

    keys = [0, s - 1] + [int(k) for k in rng.integers(0, s, 2)]
    got_kv = dkv.float().cpu().numpy().astype(np.float64)
    for j in keys:
        q_rows = np.nonzero((idx == j).any(axis=1))[0]
        assert np.all((idx[q_rows] == j).sum(axis=1) == 1)  # the lists hold distinct keys
        ref_j = np.zeros(d_qk)
        for c0 in range(0, len(q_rows), 256):
            part = q_rows[c0:c0 + 256]
            one = np.full((len(part), 1), j, dtype=np.int32)
            ref_j += _sub_bwd(x, part.tolist(), one, scale, False)["dkv"][j]
        assert rel_fro(got_kv[j], ref_j) <= TOL_GRAD_RELFRO, ("dkv", j)

    dsink_ref = np.zeros(H)
    empty = np.full((256, 1), -1, dtype=np.int32)
    for r0 in range(0, s, 256):
        dsink_ref += _sub_bwd(x, list(range(r0, r0 + 256)), empty, scale, False)["dsink"]
    assert rel_fro(dsink.cpu().numpy().astype(np.float64), dsink_ref) <= TOL_DSINK


def test_dsa_bwd_full_size_causal_sampled(attn):
    """s_q = s_kv = 4096, H = 64, QK = V = 512, top-k 2048, sink on, causal: every row's list
    is drawn from all 4096 keys, so the kernel must mask the entries after the row's own
    position.  The oracle gets each sampled row's list with those entries replaced by -1
    (its reading of an invalid entry), which is the causal computation for that row.  dQ on
    sampled rows (early rows, where most entries are masked, and late ones); dKV on sampled
    keys from the rows at or after them that list them; dSink over all rows."""
    s, H, d_qk, topk = 4096, 64, 512, 2048
    x = si.dsa_device_draws(s, s, H, d_qk, topk, False, seed=23)
    scale = d_qk ** -0.5
    x["o"], x["lse"] = _forward_inputs(x, scale, causal=True)
    dq = torch.full_like(x["q"], float("nan"))
    dkv = torch.full_like(x["kv"], float("nan"))
    dsink = torch.full_like(x["sink"], float("nan"))
    ws = torch.empty(attn.attn_dsa_bwd_workspace_size(s, d_qk), dtype=torch.uint8, device="cuda")
    attn.attn_dsa_bwd(x["q"], x["kv"], x["o"], x["do"], x["lse"], x["sink"], x["idx"], x["lens"], dq, dkv, dsink, ws,
                      scale, True)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dkv.float()).all()
    idx = x["idx"].cpu().numpy()
    later = idx > np.arange(s)[:, None]
    idx_causal = np.where(later, -1, idx).astype(np.int32)
    rng = np.random.default_rng(5)

    rows = [0, 1, 7, 130, 2047, s - 1] + [int(r) for r in rng.integers(0, s, 4)]
    ref = _sub_bwd(x, rows, idx_causal[rows], scale, False)
    got = dq[torch.as_tensor(rows, device="cuda")].float().cpu().numpy().astype(np.float64)
    for n, r in enumerate(rows):
        e = rel_fro(got[n], ref["dq"][n]) if np.any(ref["dq"][n]) else float(np.max(np.abs(got[n])))
        assert e <= TOL_GRAD_RELFRO, ("dq", r, e)

    got_kv = dkv.float().cpu().numpy().astype(np.float64)
    for j in [0, 1, s // 2, s - 1] + [int(k) for k in rng.integers(0, s, 2)]:
        q_rows = np.nonzero((idx_causal == j).any(axis=1))[0]
        ref_j = np.zeros(d_qk)
        for c0 in range(0, len(q_rows), 256):
            part = q_rows[c0:c0 + 256]
            one = np.full((len(part), 1), j, dtype=np.int32)
            ref_j += _sub_bwd(x, part.tolist(), one, scale, False)["dkv"][j]
        if np.any(ref_j):
            assert rel_fro(got_kv[j], ref_j) <= TOL_GRAD_RELFRO, ("dkv", j)
        else:
            assert np.max(np.abs(got_kv[j])) == 0.0, ("dkv of a key no row may use", j)

    dsink_ref = np.zeros(H)
    empty = np.full((256, 1), -1, dtype=np.int32)
    for r0 in range(0, s, 256):
        dsink_ref += _sub_bwd(x, list(range(r0, r0 + 256)), empty, scale, False)["dsink"]
    assert rel_fro(dsink.cpu().numpy().astype(np.float64), dsink_ref) <= TOL_DSINK
