"""Python binding of libattn_gb300.so (the C ABI declared in include/attn.h).

Argument marshalling only: every step of the forward and backward pass runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  If the
library is missing or fails to load, every call raises; there is no fallback.

Names mirror the C ABI:
    attn_fwd(q, k, v, o, lse, scale, causal, stream=None)
    attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, stream=None)
    attn_bwd_workspace_size(B, H, N, d)
    attn_fwd_layout(q, k, v, o, lse, scale, causal, layout, cu_seqlens=None, max_seqlen=None, stream=None)
    attn_bwd_layout(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, layout, ...)
    attn_bwd_layout_workspace_size(B, H, max_seqlen, d, layout, total_tokens)
    attn_decode(q, k_cache, v_cache, o, lse, workspace, scale, cache_seqlens=None, stream=None)
    attn_decode_workspace_size(B, Hq, Hkv, Nmax, d)
    attn_dsa_bwd(q, kv, o, dout, lse, sink, topk_idx, topk_len, dq, dkv, dsink, workspace, scale, causal,
                 stream=None)
    attn_dsa_bwd_workspace_size(s_kv, d_qk)
    attn_last_device_error(stream=None)
plus two allocating conveniences, ``forward`` and ``backward``.
Tensors are contiguous CUDA tensors of bfloat16 or float16: [B, H, N, d] (layout
"bhsd", the default), [B, N, H, d] ("bshd") or [total_tokens, H, d] ("packed",
with int32 device offsets cu_seqlens [B + 1]); lse is float32 [B, H, N], or
[H, total_tokens] when packed.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "AttnError", "attn_fwd", "attn_bwd", "attn_bwd_stage", "attn_bwd_workspace_size", "attn_last_device_error",
    "attn_status_string", "attn_last_launch_count", "attn_fwd_layout", "attn_bwd_layout",
    "attn_bwd_layout_workspace_size", "attn_decode", "attn_decode_workspace_size", "attn_dsa_bwd",
    "attn_dsa_bwd_workspace_size", "LAYOUTS", "forward",
    "backward", "decode", "library_path", "load",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")
_lock = threading.Lock()
_lib = None

ATTN_OK = 0
ATTN_BF16, ATTN_FP16 = 0, 1
LAYOUTS = {"bhsd": 0, "bshd": 1, "packed": 2}

EXPORTS = (
    "attn_fwd", "attn_fwd_ex", "attn_bwd_workspace_size", "attn_bwd", "attn_bwd_ex", "attn_bwd_stage",
    "attn_status_string", "attn_last_device_error", "attn_last_launch_count", "attn_fwd_layout",
    "attn_bwd_layout", "attn_bwd_layout_workspace_size", "attn_bwd_noalloc", "attn_decode",
    "attn_decode_workspace_size", "attn_dsa_bwd", "attn_dsa_bwd_workspace_size",
)


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load the library (build it first with ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with `python -m exact_attention_flashattention_gb300.build` "
                "(nvcc, sm_103a).  There is no fallback implementation.")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.attn_bwd.argtypes = [vp] * 9 + [vp, sz, i, i, i, i, f, i, vp]
        lib.attn_bwd_ex.argtypes = [vp] * 9 + [vp, sz, i, i, i, i, f, i, i, vp]
        lib.attn_bwd_stage.argtypes = [i] + [vp] * 9 + [vp, sz, i, i, i, i, f, i, i, vp]
        lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.attn_bwd_workspace_size.restype = sz
        lib.attn_fwd_layout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, i, vp]
        lib.attn_bwd_layout.argtypes = [vp] * 9 + [vp, sz, i, i, i, i, f, i, i, i, vp, i, vp]
        lib.attn_bwd_layout_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.attn_bwd_layout_workspace_size.restype = sz
        lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
        lib.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
        lib.attn_decode_workspace_size.restype = sz
        lib.attn_dsa_bwd.argtypes = [vp] * 11 + [vp, sz, i, i, i, i, i, i, f, i, vp]
        lib.attn_dsa_bwd_workspace_size.argtypes = [i, i]
        lib.attn_dsa_bwd_workspace_size.restype = sz
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_last_device_error.argtypes = [vp]
        lib.attn_last_launch_count.argtypes = []
        for fn in (lib.attn_fwd, lib.attn_fwd_ex, lib.attn_bwd, lib.attn_bwd_ex, lib.attn_bwd_stage,
                   lib.attn_fwd_layout, lib.attn_bwd_layout, lib.attn_decode, lib.attn_dsa_bwd,
                   lib.attn_last_device_error,
                   lib.attn_last_launch_count):
            fn.restype = ctypes.c_int
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16 or float16")


def _check(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None) -> None:
    """Queue the forward pass.  q, k, v, o: [B, H, N, d]; lse: float32 [B, H, N]."""
    lib = load()
    B, H, N, d = q.shape
    st = lib.attn_fwd_ex(_check(q, "q"), _check(k, "k"), _check(v, "v"), _check(o, "o"), _check(lse, "lse"),
                         B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool, stream=None) -> None:
    """Queue the backward pass.  workspace: a CUDA uint8 tensor of at least
    attn_bwd_workspace_size(B, H, N, d) bytes."""
    lib = load()
    B, H, N, d = q.shape
    st = lib.attn_bwd_ex(_check(q, "q"), _check(k, "k"), _check(v, "v"), _check(o, "o"), _check(dout, "dout"),
                         _check(lse, "lse"), _check(dq, "dq"), _check(dk, "dk"), _check(dv, "dv"),
                         _check(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                         B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")


def attn_bwd_stage(stage: int, q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool,
                   stream=None) -> None:
    """Queue one of the three backward kernels (0 preprocess, 1 main, 2 dQ convert)."""
    lib = load()
    B, H, N, d = q.shape
    st = lib.attn_bwd_stage(int(stage), _check(q, "q"), _check(k, "k"), _check(v, "v"), _check(o, "o"),
                            _check(dout, "dout"), _check(lse, "lse"), _check(dq, "dq"), _check(dk, "dk"),
                            _check(dv, "dv"), _check(workspace, "workspace"),
                            workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
                            int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, f"attn_bwd_stage({stage})")


def _layout_dims(q, layout, cu_seqlens, max_seqlen):
    """(B, H, max_seqlen, d, layout code, offsets pointer, total_tokens) of a call."""
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(LAYOUTS)}")
    if layout == "bhsd":
        B, H, N, d = q.shape
        return B, H, N, d, 0, None, 0
    if layout == "bshd":
        B, N, H, d = q.shape
        return B, H, N, d, 1, None, B * N
    import torch
    if cu_seqlens is None or max_seqlen is None:
        raise ValueError("layout 'packed' needs cu_seqlens and max_seqlen")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    total, H, d = q.shape
    return cu_seqlens.numel() - 1, H, int(max_seqlen), d, 2, _check(cu_seqlens, "cu_seqlens"), total


def attn_fwd_layout(q, k, v, o, lse, scale: float, causal: bool, layout: str, cu_seqlens=None, max_seqlen=None,
                    stream=None) -> None:
    """Queue the forward pass for a layout of LAYOUTS (tensor shapes in the module docstring)."""
    lib = load()
    B, H, N, d, lc, cu, total = _layout_dims(q, layout, cu_seqlens, max_seqlen)
    st = lib.attn_fwd_layout(_check(q, "q"), _check(k, "k"), _check(v, "v"), _check(o, "o"), _check(lse, "lse"),
                             B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), lc, cu, total,
                             _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_layout")


def attn_bwd_layout_workspace_size(B: int, H: int, max_seqlen: int, d: int, layout: str, total_tokens: int = 0) -> int:
    return int(load().attn_bwd_layout_workspace_size(B, H, max_seqlen, d, LAYOUTS[layout], total_tokens))


def attn_bwd_layout(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale: float, causal: bool, layout: str,
                    cu_seqlens=None, max_seqlen=None, stream=None) -> None:
    """Queue the backward pass for a layout of LAYOUTS."""
    lib = load()
    B, H, N, d, lc, cu, total = _layout_dims(q, layout, cu_seqlens, max_seqlen)
    st = lib.attn_bwd_layout(_check(q, "q"), _check(k, "k"), _check(v, "v"), _check(o, "o"), _check(dout, "dout"),
                             _check(lse, "lse"), _check(dq, "dq"), _check(dk, "dk"), _check(dv, "dv"),
                             _check(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                             B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), lc, cu, total,
                             _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_layout")


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, Nmax: int, d: int) -> int:
    return int(load().attn_decode_workspace_size(B, Hq, Hkv, Nmax, d))


def attn_decode(q, k_cache, v_cache, o, lse, workspace, scale: float, cache_seqlens=None, stream=None) -> None:
    """Queue decode attention.  q, o: [B, Hq, d]; k_cache, v_cache: [B, Hkv, Nmax, d];
    lse: float32 [B, Hq]; cache_seqlens: None or int32 CUDA [B]."""
    import torch
    lib = load()
    B, Hq, d = q.shape
    _, Hkv, Nmax, _ = k_cache.shape
    cu = None
    if cache_seqlens is not None:
        if cache_seqlens.dtype != torch.int32:
            raise TypeError("cache_seqlens must be int32")
        cu = _check(cache_seqlens, "cache_seqlens")
    st = lib.attn_decode(_check(q, "q"), _check(k_cache, "k_cache"), _check(v_cache, "v_cache"), _check(o, "o"),
                         _check(lse, "lse"), cu, _check(workspace, "workspace"),
                         workspace.numel() * workspace.element_size(), B, Hq, Hkv, Nmax, d, float(scale),
                         _dtype_code(q), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode")


def attn_dsa_bwd_workspace_size(s_kv: int, d_qk: int) -> int:
    return int(load().attn_dsa_bwd_workspace_size(int(s_kv), int(d_qk)))


def attn_dsa_bwd(q, kv, o, dout, lse, sink, topk_idx, topk_len, dq, dkv, dsink, workspace, scale: float,
                 causal: bool, stream=None) -> None:
    """Queue the sparse top-k attention backward (shared latent key/value rows).
    q, dq: bf16 [s_q, H, d_qk]; kv, dkv: bf16 [s_kv, d_qk]; o, dout: bf16 [s_q, H, 512];
    lse: float32 [s_q, H]; sink, dsink: float32 [H] or None; topk_idx: int32 [s_q, topk];
    topk_len: int32 [s_q] or None; workspace: at least attn_dsa_bwd_workspace_size bytes."""
    import torch
    lib = load()
    s_q, H, d_qk = q.shape
    s_kv = kv.shape[0]
    d_v = o.shape[2]
    topk = topk_idx.shape[1]
    for t, n in ((topk_idx, "topk_idx"), (topk_len, "topk_len")):
        if t is not None and t.dtype != torch.int32:
            raise TypeError(f"{n} must be int32")
    opt = lambda t, n: None if t is None else _check(t, n)
    st = lib.attn_dsa_bwd(_check(q, "q"), _check(kv, "kv"), _check(o, "o"), _check(dout, "dout"), _check(lse, "lse"),
                          opt(sink, "sink"), _check(topk_idx, "topk_idx"), opt(topk_len, "topk_len"), _check(dq, "dq"),
                          _check(dkv, "dkv"), opt(dsink, "dsink"), _check(workspace, "workspace"),
                          workspace.numel() * workspace.element_size(), s_q, s_kv, H, d_qk, d_v, topk, float(scale),
                          int(bool(causal)), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_dsa_bwd")


def attn_last_device_error(stream=None) -> int:
    return int(load().attn_last_device_error(_stream_handle(stream)))


def attn_last_launch_count() -> int:
    return int(load().attn_last_launch_count())


def forward(q, k, v, scale=None, causal=False, stream=None, layout="bhsd", cu_seqlens=None, max_seqlen=None):
    """Allocate O and L, queue the forward pass, return (O, L)."""
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    if layout == "bhsd":
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        attn_fwd(q, k, v, o, lse, scale, causal, stream)
        return o, lse
    if layout == "bshd":
        B, N, H, _ = q.shape
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    attn_fwd_layout(q, k, v, o, lse, scale, causal, layout, cu_seqlens, max_seqlen, stream)
    return o, lse


def backward(q, k, v, o, dout, lse, scale=None, causal=False, workspace=None, stream=None, layout="bhsd",
             cu_seqlens=None, max_seqlen=None):
    """Allocate dQ, dK, dV (and the workspace if not given), queue the backward pass."""
    import torch
    B, H, N, d, _, _, total = _layout_dims(q, layout, cu_seqlens, max_seqlen)
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(attn_bwd_layout_workspace_size(B, H, N, d, layout, total), dtype=torch.uint8,
                                device=q.device)
    if layout == "bhsd":
        attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, stream)
    else:
        attn_bwd_layout(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, causal, layout, cu_seqlens, max_seqlen,
                        stream)
    return dq, dk, dv


def decode(q, k_cache, v_cache, cache_seqlens=None, scale=None, workspace=None, stream=None):
    """Allocate O, L (and the workspace if not given), queue decode attention, return (O, L)."""
    import torch
    B, Hq, d = q.shape
    _, Hkv, Nmax, _ = k_cache.shape
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, Hq, Hkv, Nmax, d), dtype=torch.uint8, device=q.device)
    attn_decode(q, k_cache, v_cache, o, lse, workspace, scale, cache_seqlens, stream)
    return o, lse
