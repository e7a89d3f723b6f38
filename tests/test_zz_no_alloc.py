"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a serving engine that owns one pre-sized memory pool, a plugin host
that hands its plugins only their inputs and outputs, code that cannot accept
cudaMalloc's implicit synchronisation) get a backward whose scratch is a fixed
array inside the library.  These tests call it through the C ABI, twice in a
row, and check its results against the workspace entry point attn_bwd within
the parity tolerance and against the FP64 oracle directly; check that the
device's free memory does not change across the second call (the array was
reserved by the first); and check that a problem too large for the fixed array
is refused before anything is queued.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math
import os

import numpy as np
import pytest

import oracle
from attn_cases import TOL_GRAD_RELFRO, f64, input_bits, rel_fro, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATTN_ERR_WORKSPACE = 4
SCRATCH_BYTES = 64 << 20


@pytest.fixture(scope="module")
def lib():
    import exact_attention_flashattention_gb300 as attn
    from exact_attention_flashattention_gb300 import build
    if not os.path.exists(attn.library_path()):
        build.build()
    lib = attn.load()
    fn = lib.attn_bwd_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp] * 9 + [i, i, i, i, f, i, i, vp]
    fn.restype = ctypes.c_int
    return attn, lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("B,H,N,d,causal,dtype", [(1, 4, 1024, 128, True, "bf16"), (2, 2, 512, 64, False, "fp16")])
def test_noalloc_matches_workspace_entry_point(lib, B, H, N, d, causal, dtype):
    attn, clib = lib
    assert attn.attn_bwd_workspace_size(B, H, N, d) <= SCRATCH_BYTES
    bits = input_bits(314 + N + d, B * H, N, d, dtype)
    q, k, v, do = (to_device(bits[n], B, H, dtype) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = attn.forward(q, k, v, scale, causal)
    ref = [to_f64(t) for t in attn.backward(q, k, v, o, do, lse, scale, causal)]
    shp = (B, H, N, d)
    exact = oracle.attn_bwd(*(f64(bits[n], dtype).reshape(shp) for n in ("q", "k", "v", "do")), scale, causal)
    code = 0 if dtype == "bf16" else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = clib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, H, N, d, scale, int(causal), code, stream)
        assert st == 0, attn.attn_status_string(st)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert attn.attn_last_device_error() == 0
        if call == 1:
            # the scratch array was reserved with the first call's module load; later calls reserve nothing
            assert free_after == free_before, (free_before, free_after)
        for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g = to_f64(got)
            assert np.isfinite(g).all(), (call, name)
            e = rel_fro(g, r)
            assert e <= TOL_GRAD_RELFRO, (call, name, "vs attn_bwd", e)
            e = rel_fro(g, exact[name])
            assert e <= TOL_GRAD_RELFRO, (call, name, "vs the oracle", e)


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    attn, clib = lib
    B, H, N, d = 8, 16, 4096, 128
    assert attn.attn_bwd_workspace_size(B, H, N, d) > SCRATCH_BYTES
    p = ctypes.c_void_p(256)  # never dereferenced: the call is refused first
    st = clib.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0.1, 1, 0, ctypes.c_void_p(0))
    assert st == ATTN_ERR_WORKSPACE
    assert clib.attn_last_launch_count() == 0
