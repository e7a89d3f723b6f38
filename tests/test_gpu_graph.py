"""The forward and backward captured once in a CUDA graph and replayed.

The library allocates nothing, so a capture of attn_fwd + attn_bwd (4 kernels)
replays on new inputs copied into the same buffers.  With packed sequences the
forward and the backward's main kernel also zero their work counters (words of
the library's own device array) inside the capture, so each replay distributes
the work afresh.  Replays must give exactly the eager results for O, L, dK and dV (dQ
adds FP32 partials in no fixed order: compared within the cross-path bound of
the layout tests), and still match the FP64 oracle.
"""
import math

import numpy as np
import pytest

import oracle
from attn_cases import TOL_GRAD_RELFRO, TOL_L_MAXABS, TOL_O_MAXABS, f64, input_bits, rel_fro, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_graph_replay_matches_eager_and_oracle():
    import exact_attention_flashattention_gb300 as attn
    attn.load()
    B, H, N, d, causal, dtype = 1, 4, 640, 128, True, "bf16"
    scale = 1.0 / math.sqrt(d)
    shape = (B, H, N, d)
    bufs = {n: torch.empty(shape, dtype=torch.bfloat16, device="cuda") for n in ("q", "k", "v", "do")}
    o, dq, dk, dv = (torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

    def step(stream):
        attn.attn_fwd(bufs["q"], bufs["k"], bufs["v"], o, lse, scale, causal, stream)
        attn.attn_bwd(bufs["q"], bufs["k"], bufs["v"], o, bufs["do"], lse, dq, dk, dv, ws, scale, causal, stream)

    def load_inputs(seed):
        x = input_bits(seed, B * H, N, d, dtype)
        for n in bufs:
            bufs[n].copy_(to_device(x[n], B, H, dtype))
        return x

    stream = torch.cuda.Stream()
    load_inputs(1)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step(stream)                          # warm-up outside the capture (first-call set-up)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()

    for seed in (2, 3):
        x = load_inputs(seed)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert attn.attn_last_device_error() == 0
        got = dict(o=to_f64(o), lse=to_f64(lse), dq=to_f64(dq), dk=to_f64(dk), dv=to_f64(dv))
        with torch.cuda.stream(stream):
            step(stream)
        stream.synchronize()
        eager = dict(o=to_f64(o), lse=to_f64(lse), dq=to_f64(dq), dk=to_f64(dk), dv=to_f64(dv))
        for n in ("o", "lse", "dk", "dv"):
            assert np.array_equal(got[n], eager[n]), n
        assert rel_fro(got["dq"], eager["dq"]) <= 2e-3
        ref = oracle.attn_bwd(*(f64(x[n], dtype) for n in ("q", "k", "v", "do")), scale, causal)
        assert np.max(np.abs(got["o"] - ref["o"].reshape(shape))) <= TOL_O_MAXABS
        assert np.max(np.abs(got["lse"] - ref["lse"].reshape(B, H, N))) <= TOL_L_MAXABS
        for n in ("dq", "dk", "dv"):
            assert rel_fro(got[n], ref[n].reshape(shape)) <= TOL_GRAD_RELFRO, n


def test_packed_graph_replay():
    """Packed sequences, more units than SMs: each CTA of the forward and of the backward's
    main kernel takes several units from its launch's work counter.  Replays (and an eager
    call between them) give the eager O, L, dK and dV bit for bit and dQ within the cross-path
    bound, and match the oracle sequence by sequence."""
    import exact_attention_flashattention_gb300 as attn
    attn.load()
    lens, H, d, causal, dtype = [1000, 40, 700, 3000], 8, 128, True, "bf16"
    scale = 1.0 / math.sqrt(d)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, max_seqlen = int(cu[-1]), max(lens)
    q, k, v, do = (torch.empty((total, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((H, total), dtype=torch.float32, device="cuda")
    cu_dev = torch.from_numpy(cu).to("cuda")
    ws = torch.empty(attn.attn_bwd_layout_workspace_size(len(lens), H, max_seqlen, d, "packed", total),
                     dtype=torch.uint8, device="cuda")

    def step(stream):
        attn.attn_fwd_layout(q, k, v, o, lse, scale, causal, "packed", cu_dev, max_seqlen, stream)
        attn.attn_bwd_layout(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, "packed", cu_dev, max_seqlen,
                             stream)

    def load_inputs(seed):
        slices = [input_bits(seed * 100 + b, H, n, d, dtype) for b, n in enumerate(lens)]
        for t, name in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
            arr = np.concatenate([x[name].transpose(1, 0, 2) for x in slices])   # [H, n, d] -> [n, H, d]
            t.copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16))
        return slices

    def snapshot():
        return dict(o=to_f64(o), lse=to_f64(lse), dq=to_f64(dq), dk=to_f64(dk), dv=to_f64(dv))

    stream = torch.cuda.Stream()
    load_inputs(1)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()

    for seed in (2, 3):
        slices = load_inputs(seed)
        torch.cuda.synchronize()
        graph.replay()
        graph.replay()
        torch.cuda.synchronize()
        assert attn.attn_last_device_error() == 0
        got = snapshot()
        with torch.cuda.stream(stream):
            step(stream)
        stream.synchronize()
        eager = snapshot()
        for n in ("o", "lse", "dk", "dv"):
            assert np.array_equal(got[n], eager[n]), n
        assert rel_fro(got["dq"], eager["dq"]) <= 2e-3
        for b, x in enumerate(slices):
            rows = slice(cu[b], cu[b + 1])
            ref = oracle.attn_bwd(*(f64(x[n], dtype) for n in ("q", "k", "v", "do")), scale, causal)
            assert np.max(np.abs(got["o"][rows].transpose(1, 0, 2) - ref["o"])) <= TOL_O_MAXABS, b
            assert np.max(np.abs(got["lse"][:, rows] - ref["lse"])) <= TOL_L_MAXABS, b
            for n in ("dq", "dk", "dv"):
                assert rel_fro(got[n][rows].transpose(1, 0, 2), ref[n]) <= TOL_GRAD_RELFRO, (b, n)
