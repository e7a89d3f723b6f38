"""Decode attention (one query per head against a key/value cache) vs the FP64 oracle.

The oracle's row entry point gives the reference: for batch b and query head h,
the row of a query matrix whose row 0 is q[b, h] over the cache's first len_b
keys, non-causal (every cached key is visible), which is the decode output.
Cases cover grouped queries (G = Hq / Hkv from 1 to 128, i.e. one to all four
softmax warps), d = 64 and 128, bf16 and fp16, cache lengths of 0, 1, ragged and
full, several key chunks (1024 keys at d = 128, 2048 at d = 64), and more work items than SMs.  Tolerances as for
the forward: O max-abs 1e-2, L max-abs 1e-3.  Outputs are pre-filled with NaN.
"""
import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from attn_cases import TOL_L_MAXABS, TOL_O_MAXABS, f64, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, Nmax, d, dtype, cache lengths (None: all Nmax)
    (2, 8, 2, 1000, 128, "bf16", [1000, 513]),
    (3, 4, 4, 300, 64, "fp16", None),
    (1, 16, 1, 2500, 128, "bf16", [2500]),
    (4, 2, 2, 700, 64, "bf16", [0, 1, 129, 700]),
    (1, 64, 1, 300, 64, "bf16", None),
    (1, 128, 1, 200, 128, "bf16", None),
    (16, 32, 8, 3000, 128, "bf16", None),      # 128 groups x 3 chunks: more items than SMs
    (2, 8, 4, 5000, 64, "fp16", [5000, 2049]),  # d = 64: three 2048-key chunks, one of them a single key
]


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _dev(bits, shape, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).reshape(shape).to("cuda")
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def _inputs(seed, B, Hq, Hkv, Nmax, d, dtype):
    qb = si.tensor_heads(seed, "q", B * Hq, 1, d, 1.0, dtype)          # [B Hq, 1, d]
    kb = si.tensor_heads(seed, "k", B * Hkv, Nmax, d, 1.0, dtype)      # [B Hkv, Nmax, d]
    vb = si.tensor_heads(seed, "v", B * Hkv, Nmax, d, 1.0, dtype)
    return qb, kb, vb


def _reference(qb, kb, vb, B, Hq, Hkv, d, lens, dtype, scale):
    G = Hq // Hkv
    o = np.zeros((B, Hq, d))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        n = lens[b]
        if n == 0:
            continue
        for h in range(Hq):
            kv = b * Hkv + h // G
            qfull = np.zeros((n, d))
            qfull[0] = f64(qb[b * Hq + h, 0], dtype)
            o_r, l_r, _ = oracle.attn_rows(qfull, f64(kb[kv, :n], dtype), f64(vb[kv, :n], dtype),
                                           np.array([0], dtype=np.int64), scale, False)
            o[b, h], lse[b, h] = o_r[0], l_r[0]
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,Nmax,d,dtype,lens", CASES)
def test_decode_matches_oracle(attn, B, Hq, Hkv, Nmax, d, dtype, lens):
    scale = 1.0 / math.sqrt(d)
    qb, kb, vb = _inputs(7000 + Nmax + d + Hq, B, Hq, Hkv, Nmax, d, dtype)
    q = _dev(qb, (B, Hq, d), dtype)
    k = _dev(kb, (B, Hkv, Nmax, d), dtype)
    v = _dev(vb, (B, Hkv, Nmax, d), dtype)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_decode_workspace_size(B, Hq, Hkv, Nmax, d), dtype=torch.uint8, device="cuda")
    seq = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    attn.attn_decode(q, k, v, o, lse, ws, scale, seq)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    got_o, got_l = to_f64(o), to_f64(lse)
    lens = [Nmax] * B if lens is None else lens
    ref_o, ref_l = _reference(qb, kb, vb, B, Hq, Hkv, d, lens, dtype, scale)
    assert np.isfinite(got_o).all(), "unwritten or non-finite O"
    assert np.max(np.abs(got_o - ref_o)) <= TOL_O_MAXABS
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got_l[b] == -np.inf) and np.all(got_o[b] == 0.0)
        else:
            assert np.max(np.abs(got_l[b] - ref_l[b])) <= TOL_L_MAXABS, b


def test_decode_bad_cache_lengths_are_reported(attn):
    """A cache length outside [0, Nmax] is treated as 0 (nothing of that batch is read) and
    reported through the device error word; the other batches are unaffected."""
    B, Hq, Hkv, Nmax, d, dtype = 3, 2, 1, 256, 64, "bf16"
    scale = 1.0 / math.sqrt(d)
    qb, kb, vb = _inputs(7777, B, Hq, Hkv, Nmax, d, dtype)
    q, k, v = _dev(qb, (B, Hq, d), dtype), _dev(kb, (B, Hkv, Nmax, d), dtype), _dev(vb, (B, Hkv, Nmax, d), dtype)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_decode_workspace_size(B, Hq, Hkv, Nmax, d), dtype=torch.uint8, device="cuda")
    attn.attn_decode(q, k, v, o, lse, ws, scale, torch.tensor([100, -3, Nmax + 1], dtype=torch.int32, device="cuda"))
    assert attn.attn_last_device_error() == 1          # ATTN_ERR_INVALID_ARG
    got_o, got_l = to_f64(o), to_f64(lse)
    assert np.all(got_o[1:] == 0.0) and np.all(got_l[1:] == -np.inf)
    ref_o, ref_l = _reference(qb, kb, vb, B, Hq, Hkv, d, [100, 0, 0], dtype, scale)
    assert np.max(np.abs(got_o[0] - ref_o[0])) <= TOL_O_MAXABS
    assert np.max(np.abs(got_l[0] - ref_l[0])) <= TOL_L_MAXABS


@pytest.mark.parametrize("B,Hq,Hkv,Nmax,d,launches", [
    (2, 8, 2, 1000, 128, 1),    # one chunk per (batch, KV head): the chunk kernel writes O and L
    (1, 16, 1, 2500, 128, 2),   # one group, three chunks: chunk kernel, then the combination
])
def test_decode_single_chunk_and_split_paths(attn, B, Hq, Hkv, Nmax, d, launches):
    """Both ways a decode call ends, each against the oracle: with one key chunk per group the
    chunk kernel's normalised O and L are the results (one launch); with several, a second
    kernel combines the chunks."""
    dtype = "bf16"
    scale = 1.0 / math.sqrt(d)
    qb, kb, vb = _inputs(8100 + Nmax, B, Hq, Hkv, Nmax, d, dtype)
    q, k, v = _dev(qb, (B, Hq, d), dtype), _dev(kb, (B, Hkv, Nmax, d), dtype), _dev(vb, (B, Hkv, Nmax, d), dtype)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_decode_workspace_size(B, Hq, Hkv, Nmax, d), dtype=torch.uint8, device="cuda")
    attn.attn_decode(q, k, v, o, lse, ws, scale, None)
    assert attn.attn_last_launch_count() == launches
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0
    ref_o, ref_l = _reference(qb, kb, vb, B, Hq, Hkv, d, [Nmax] * B, dtype, scale)
    assert np.max(np.abs(to_f64(o) - ref_o)) <= TOL_O_MAXABS
    assert np.max(np.abs(to_f64(lse) - ref_l)) <= TOL_L_MAXABS
