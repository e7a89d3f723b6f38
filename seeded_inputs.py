"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no attention arithmetic: it only draws numbers.  Both the
tests (oracle side) and the CUDA binding side get their Q, K, V, dO from here,
so that the two are fed the same rounded values.

Generator (counter-based, every element independent of how many others are
drawn, so a single head can be regenerated alone):

* SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output_n = mix(key + (n + 1) * 0x9E3779B97F4A7C15)
  with the published 64-bit finaliser ``mix``.
* Two outputs per pair -> two doubles in (0, 1] from their top 53 bits ->
  Box-Muller (G. Box, M. Muller 1958): r = sqrt(-2 ln u1), angles 2 pi u2.
* float32 sample * sigma, then round-to-nearest-even to bfloat16 or float16.

The per-head key is mix(base_seed ^ mix(tensor_id * 2^32 + head)), so head h of
tensor t is the same whichever subset of heads is drawn.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "do": 4, "kv": 5, "sink": 6, "idx": 7}


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(x: int) -> int:
    with np.errstate(over="ignore"):
        return int(_mix(np.array([x & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def head_key(base_seed: int, tensor_id: int, head: int) -> int:
    inner = _mix_scalar((tensor_id << 32) + head)
    return _mix_scalar((base_seed & 0xFFFFFFFFFFFFFFFF) ^ inner)


def splitmix64_stream(key: int, n: int) -> np.ndarray:
    """First n outputs of the SplitMix64 stream with the given key."""
    with np.errstate(over="ignore"):
        ctr = np.arange(1, n + 1, dtype=np.uint64)
        return _mix(np.uint64(key) + ctr * GAMMA)


def standard_normal(key: int, n: int) -> np.ndarray:
    """n float32 standard-normal samples from one SplitMix64 stream."""
    m = (n + 1) // 2
    bits = splitmix64_stream(key, 2 * m)
    # top 53 bits -> (0, 1]: (k + 1) / 2^53
    u = ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n].astype(np.float32)


def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_fp16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> float16 bit patterns (numpy's cast rounds to nearest even)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16_bits(x)
    if dtype == "fp16":
        return round_fp16_bits(x)
    raise ValueError(dtype)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(b)
    if dtype == "fp16":
        return fp16_bits_to_f32(b)
    raise ValueError(dtype)


def tensor_heads(base_seed: int, name: str, BH: int, N: int, d: int, sigma: float,
                 dtype: str = "bf16", heads=None, threads: int | None = None) -> np.ndarray:
    """16-bit patterns [len(heads), N, d] of tensor `name` for the given heads
    (default: all BH heads), entries ~ N(0, sigma^2) rounded to `dtype`."""
    if heads is None:
        heads = range(BH)
    heads = list(heads)
    tid = TENSOR_IDS[name]
    out = np.empty((len(heads), N, d), dtype=np.uint16)

    def one(ix):
        h = heads[ix]
        z = standard_normal(head_key(base_seed, tid, h), N * d) * np.float32(sigma)
        out[ix] = to_bits(z, dtype).reshape(N, d)

    nthr = threads or min(len(heads), os.cpu_count() or 1, 16)
    if nthr <= 1 or len(heads) <= 1:
        for ix in range(len(heads)):
            one(ix)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, range(len(heads))))
    return out


def late_spike(q_bits: np.ndarray, k_bits: np.ndarray, dtype: str, alpha: float,
               rows, tile: int = 128) -> np.ndarray:
    """Adversarial 'late spike' keys for one head (q_bits, k_bits: [N, d]).

    For each query row i in `rows`, key (last tile start + i mod tile) is set to
    alpha * q_i / |q_i|, so that row's largest score arrives in the final key
    tile.  Returns new key bits [N, d]."""
    q = bits_to_f32(q_bits, dtype).astype(np.float64)
    k = bits_to_f32(k_bits, dtype).astype(np.float32).copy()
    N = q.shape[0]
    last = ((N - 1) // tile) * tile
    for i in rows:
        j = last + (i % tile)
        if j >= N:
            j = N - 1
        nrm = np.linalg.norm(q[i]) or 1.0
        k[j] = (alpha * q[i] / nrm).astype(np.float32)
    return to_bits(k, dtype)


def _rows_normal(base_seed: int, name: str, rows, width: int, sigma: float) -> np.ndarray:
    """float32 [len(rows), width]: row r drawn from its own stream (so one row can be
    regenerated alone), entries ~ N(0, sigma^2)."""
    tid = TENSOR_IDS[name]
    out = np.empty((len(rows), width), dtype=np.float32)
    for ix, r in enumerate(rows):
        out[ix] = standard_normal(head_key(base_seed, tid, int(r)), width) * np.float32(sigma)
    return out


def topk_indices(base_seed: int, s_q: int, s_kv: int, topk: int, causal: bool, rows=None):
    """Key index lists of a sparse top-k attention: for query i, min(topk, n_i) distinct
    keys in random order, n_i = i + 1 when causal (keys 0..i) else s_kv, padded with -1.
    Returns (idx int32 [len(rows), topk], lengths int32 [len(rows)]).  Each row is a
    random permutation (keys sorted by a SplitMix64 draw), so rows are independent."""
    rows = range(s_q) if rows is None else rows
    rows = list(rows)
    tid = TENSOR_IDS["idx"]
    idx = np.full((len(rows), topk), -1, dtype=np.int32)
    lens = np.empty(len(rows), dtype=np.int32)
    for ix, i in enumerate(rows):
        n = min(int(i) + 1, s_kv) if causal else s_kv
        keys = splitmix64_stream(head_key(base_seed, tid, int(i)), n)
        take = np.argsort(keys, kind="stable")[:min(topk, n)]
        idx[ix, :take.shape[0]] = take.astype(np.int32)
        lens[ix] = take.shape[0]
    return idx, lens


def dsa_inputs(base_seed: int, s_q: int, s_kv: int, H: int, d_qk: int, d_v: int, topk: int,
               causal: bool, sigma: float = 1.0, rows=None, with_kv: bool = True) -> dict:
    """Synthetic inputs of a sparse top-k attention with one shared latent key/value row
    per key (bf16 bit patterns unless noted):
      q [n, H, d_qk], do [n, H, d_v] for the query rows `rows` (default all s_q),
      kv [s_kv, d_qk] (if with_kv), sink float32 [H], idx int32 [n, topk], lens int32 [n].
    Values ~ N(0, sigma^2) for q, kv, do; sink ~ N(0, 1)."""
    rows = list(range(s_q) if rows is None else rows)
    out = {}
    out["q"] = round_bf16_bits(_rows_normal(base_seed, "q", rows, H * d_qk, sigma)).reshape(len(rows), H, d_qk)
    out["do"] = round_bf16_bits(_rows_normal(base_seed, "do", rows, H * d_v, sigma)).reshape(len(rows), H, d_v)
    if with_kv:
        out["kv"] = round_bf16_bits(_rows_normal(base_seed, "kv", range(s_kv), d_qk, sigma))
    out["sink"] = standard_normal(head_key(base_seed, TENSOR_IDS["sink"], 0), H)
    out["idx"], out["lens"] = topk_indices(base_seed, s_q, s_kv, topk, causal, rows)
    return out


def dsa_device_draws(s_q: int, s_kv: int, H: int, d_qk: int, topk: int, causal: bool, seed: int = 17,
                     d_v: int = 512, device: str = "cuda") -> dict:
    """Sparse top-k attention inputs drawn on the GPU with torch's generator, for sizes where
    the host generator above is too slow (full-size timing and sampled checks): q [s_q, H,
    d_qk], kv [s_kv, d_qk], do [s_q, H, d_v] ~ N(0, 1) rounded to bf16; sink [H] ~ N(0, 1)
    float32; each row's list = min(topk, n_i) distinct random keys (keys 0..i when causal,
    n_i = i + 1, else s_kv), padded with -1; lens [s_q] the list lengths.  Draws only: the
    forward's O and L, which the backward also takes, are for the caller to compute."""
    import torch
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    q = torch.randn((s_q, H, d_qk), generator=g, device=dev).to(torch.bfloat16)
    kv = torch.randn((s_kv, d_qk), generator=g, device=dev).to(torch.bfloat16)
    do = torch.randn((s_q, H, d_v), generator=g, device=dev).to(torch.bfloat16)
    sink = torch.randn((H,), generator=g, device=dev)
    idx = torch.empty((s_q, topk), dtype=torch.int32, device=dev)
    lens = torch.empty((s_q,), dtype=torch.int32, device=dev)
    for r0 in range(0, s_q, 512):
        r1 = min(s_q, r0 + 512)
        keys = torch.rand((r1 - r0, s_kv), generator=g, device=dev)
        rows = torch.arange(r0, r1, device=dev)[:, None]
        if causal:
            keys = torch.where(torch.arange(s_kv, device=dev)[None, :] <= rows, keys, torch.full_like(keys, 2.0))
        order = keys.argsort(dim=1)[:, :topk].to(torch.int32)
        if causal:
            n = torch.clamp(rows[:, 0] + 1, max=min(topk, s_kv))
        else:
            n = torch.full((r1 - r0,), min(topk, s_kv), device=dev)
        pos = torch.arange(topk, device=dev)[None, :]
        idx[r0:r1] = torch.where(pos < n[:, None], order, torch.full_like(order, -1))
        lens[r0:r1] = n.to(torch.int32)
    return dict(q=q, kv=kv, do=do, sink=sink, idx=idx, lens=lens)
