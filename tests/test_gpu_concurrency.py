"""Calls on different streams do not interfere.

The library keeps a little device state of its own: the error word and the per-launch work
counters that packed sequences and causal work take units from.  Two unrelated problems, one of
packed causal sequences and one fixed-length fp16 problem, are run forward and backward
back to back on one stream, then again interleaved on two streams, three times over.  The
interleaved results must equal the sequential ones: O, L, dK and dV bit for bit (their
arithmetic order is fixed), dQ to the rounding of its FP32 accumulation order (the partials
of different key tiles arrive in a nondeterministic order).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import exact_attention_flashattention_gb300 as a
    a.load()
    return a


def _problem(attn, kind, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if kind == "packed":
        lens = [300, 1000, 129, 2048, 0, 777]
        H, d, dt = 8, 128, torch.bfloat16
        total = sum(lens)
        shape = (total, H, d)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
        spec = dict(layout="packed", cu=cu, maxlen=max(lens), B=len(lens), H=H, d=d, total=total,
                    lse_shape=(H, total))
    else:
        B, H, N, d, dt = 2, 8, 1536, 64, torch.float16
        shape = (B, H, N, d)
        spec = dict(layout="bhsd", cu=None, maxlen=N, B=B, H=H, d=d, total=0, lse_shape=(B, H, N))
    t = {n: torch.randn(shape, generator=g, device="cuda").to(dt) for n in ("q", "k", "v", "do")}
    spec["inputs"] = t
    spec["ws_bytes"] = attn.attn_bwd_layout_workspace_size(spec["B"], spec["H"], spec["maxlen"], spec["d"],
                                                           spec["layout"], spec["total"])
    return spec


def _buffers(spec):
    q = spec["inputs"]["q"]
    return dict(o=torch.empty_like(q), lse=torch.empty(spec["lse_shape"], device="cuda"),
                dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q),
                ws=torch.empty(spec["ws_bytes"], dtype=torch.uint8, device="cuda"))


def _run(attn, spec, buf, stream):
    t = spec["inputs"]
    sc = 1.0 / math.sqrt(spec["d"])
    attn.attn_fwd_layout(t["q"], t["k"], t["v"], buf["o"], buf["lse"], sc, True, spec["layout"], spec["cu"],
                         spec["maxlen"], stream)
    attn.attn_bwd_layout(t["q"], t["k"], t["v"], buf["o"], t["do"], buf["lse"], buf["dq"], buf["dk"], buf["dv"],
                         buf["ws"], sc, True, spec["layout"], spec["cu"], spec["maxlen"], stream)


def test_two_streams_match_one(attn):
    specs = [_problem(attn, "packed", 1), _problem(attn, "bhsd", 2)]
    ref = [_buffers(s) for s in specs]
    main = torch.cuda.current_stream()
    for s, b in zip(specs, ref):
        _run(attn, s, b, main)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = [_buffers(s) for s in specs]
    for _ in range(3):
        for s, b, st in zip(specs, got, streams):
            _run(attn, s, b, st)
    torch.cuda.synchronize()
    assert attn.attn_last_device_error() == 0

    for s, r, g in zip(specs, ref, got):
        for name in ("o", "lse", "dk", "dv"):
            assert torch.equal(r[name], g[name]), (s["layout"], name)
        a, b = r["dq"].float(), g["dq"].float()
        err = float((a - b).norm() / a.norm())
        assert err <= 1e-5, (s["layout"], "dq", err)
