"""The C-ABI library loads and exports every symbol include/attn.h declares;
argument checks that run before any CUDA call return the documented codes.
No kernel is launched here (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    import shutil
    from exact_attention_flashattention_gb300 import build as b
    if not os.path.exists(b.LIB):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build the library")
        b.build()
    import exact_attention_flashattention_gb300 as attn
    return attn.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_ex", "attn_bwd", "attn_bwd_ex", "attn_bwd_workspace_size",
              "attn_status_string", "attn_last_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_names_match_exports():
    import exact_attention_flashattention_gb300 as attn
    assert set(attn.EXPORTS) <= set(declared_functions())


def test_argument_checks_before_any_launch(lib):
    import exact_attention_flashattention_gb300 as attn
    vp = ctypes.c_void_p
    p = vp(256)  # never dereferenced: every case below is rejected first
    null = vp(0)
    assert lib.attn_fwd(null, p, p, p, p, 1, 1, 128, 128, 1.0, 1, null) == 1          # INVALID_ARG
    assert lib.attn_fwd(p, p, p, p, p, 1, 1, 128, 96, 1.0, 1, null) == 2              # d unsupported
    assert lib.attn_fwd(p, p, p, p, p, 1, 1, 0, 128, 1.0, 1, null) == 1               # N <= 0
    assert lib.attn_fwd(p, p, p, p, p, 1 << 15, 1 << 15, 256, 128, 1.0, 1, null) == 2  # too large
    assert lib.attn_fwd(p, p, p, p, p, 0, 1, 128, 128, 1.0, 1, null) == 1             # B <= 0
    assert lib.attn_fwd(vp(258), p, p, p, p, 1, 1, 128, 128, 1.0, 1, null) == 3       # alignment
    assert lib.attn_fwd_ex(p, p, p, p, p, 1, 1, 128, 128, 1.0, 1, 7, null) == 1       # bad dtype
    ws = attn.attn_bwd_workspace_size(1, 1, 128, 128)
    assert ws >= 128 * 4 * 2 + 128 * 128 * 4 and ws % 256 == 0
    # any N: the workspace rows are padded to whole 128-row tiles
    assert attn.attn_bwd_workspace_size(1, 1, 100, 128) == attn.attn_bwd_workspace_size(1, 1, 128, 128)
    assert attn.attn_bwd_workspace_size(1, 1, 129, 64) == attn.attn_bwd_workspace_size(1, 1, 256, 64)
    assert attn.attn_bwd_workspace_size(1, 1, 0, 64) == 0
    assert lib.attn_bwd(p, p, p, p, p, p, p, p, p, null, 0, 1, 1, 128, 128, 1.0, 1, null) == 4   # workspace
    assert lib.attn_bwd(p, p, p, p, p, p, p, p, p, vp(512), ws - 1, 1, 1, 128, 128, 1.0, 1, null) == 4
    assert lib.attn_bwd(p, p, p, p, p, p, p, p, p, vp(512 + 16), ws, 1, 1, 128, 128, 1.0, 1, null) == 3
    assert lib.attn_last_launch_count() == 0
    for s in range(7):
        assert attn.attn_status_string(s).startswith("ATTN_")


def test_layout_argument_checks_before_any_launch(lib):
    import exact_attention_flashattention_gb300 as attn
    vp = ctypes.c_void_p
    p = vp(256)  # never dereferenced: every case below is rejected (or has nothing to do) first
    null = vp(0)
    cu = vp(4096)
    BHSD, BSHD, PACKED = 0, 1, 2
    f = lib.attn_fwd_layout
    assert f(p, p, p, p, p, 1, 1, 128, 128, 1.0, 1, 0, 7, null, 0, null) == 1         # unknown layout
    assert f(p, p, p, p, p, 2, 1, 128, 128, 1.0, 1, 0, PACKED, null, 256, null) == 1  # packed needs offsets
    assert f(p, p, p, p, p, 2, 1, 128, 128, 1.0, 1, 0, BSHD, cu, 256, null) == 1      # offsets only when packed
    assert f(p, p, p, p, p, 2, 1, 128, 128, 1.0, 1, 0, PACKED, vp(4098), 256, null) == 3  # offsets alignment
    assert f(p, p, p, p, p, 2, 1, 128, 128, 1.0, 1, 0, PACKED, cu, -1, null) == 1     # negative token count
    assert f(p, p, p, p, p, 2, 1, 128, 96, 1.0, 1, 0, PACKED, cu, 256, null) == 2     # d unsupported
    assert f(p, p, p, p, vp(260), 2, 1, 128, 128, 1.0, 1, 0, BSHD, null, 0, null) == 3  # alignment
    # packed with no tokens at all: nothing to do, nothing queued, no CUDA call
    assert f(p, p, p, p, p, 2, 1, 128, 128, 1.0, 1, 0, PACKED, cu, 0, null) == 0
    assert lib.attn_last_launch_count() == 0
    ws = attn.attn_bwd_layout_workspace_size
    # fixed-length layouts: the same rows as attn_bwd_workspace_size
    assert ws(2, 3, 300, 64, "bshd", 0) == attn.attn_bwd_workspace_size(2, 3, 300, 64)
    assert ws(2, 3, 300, 64, "bhsd", 0) == attn.attn_bwd_workspace_size(2, 3, 300, 64)
    # packed: per head 128 (ceil(tokens / 128) + B) rows (each sequence padded to whole tiles,
    # starting on a 128-row boundary)
    rows = 2 * 128 * (4 + 3)
    up = lambda x: (x + 255) // 256 * 256
    lse2 = up(rows * 4)
    dq = up(lse2 + rows * 4)
    assert ws(3, 2, 300, 64, "packed", 500) == up(dq + rows * 64 * 4)
    assert ws(3, 2, 300, 64, "packed", -1) == 0
    assert lib.attn_bwd_layout(p, p, p, p, p, p, p, p, p, null, 0, 3, 2, 300, 64, 1.0, 1, 0, PACKED, cu, 500,
                               null) == 4                                            # workspace
    assert lib.attn_last_launch_count() == 0


def test_decode_argument_checks_before_any_launch(lib):
    import exact_attention_flashattention_gb300 as attn
    vp = ctypes.c_void_p
    p = vp(256)
    null = vp(0)
    d = lib.attn_decode
    wsz = attn.attn_decode_workspace_size
    # sized for the finest split, chunks of 1024 keys at d = 128 (2048 at d = 64; a launch may use
    # longer ones); per (group, chunk, query head): d FP32 values and one L
    rows = 2 * 2 * 3 * 4                    # B Hkv, 3 chunks of 3000 keys, G = 4
    up = lambda x: (x + 255) // 256 * 256
    assert wsz(2, 8, 2, 3000, 128) == up(up(rows * 128 * 4) + rows * 4)
    assert wsz(2, 6, 4, 3000, 128) == 0      # Hq not a multiple of Hkv
    assert wsz(1, 256, 1, 100, 64) == 0      # G > 128
    assert wsz(1, 4, 4, 100, 96) == 0        # d unsupported
    n = wsz(2, 8, 2, 1000, 128)
    assert d(null, p, p, p, p, null, p, n, 2, 8, 2, 1000, 128, 1.0, 0, null) == 1          # null q
    assert d(p, p, p, p, p, null, p, n, 2, 6, 4, 1000, 128, 1.0, 0, null) == 1             # Hq % Hkv
    assert d(p, p, p, p, p, null, p, n, 2, 8, 2, 1000, 96, 1.0, 0, null) == 2              # d unsupported
    assert d(p, p, p, p, p, null, null, 0, 2, 8, 2, 1000, 128, 1.0, 0, null) == 4          # workspace
    assert d(p, p, p, p, p, null, vp(512), n - 1, 2, 8, 2, 1000, 128, 1.0, 0, null) == 4   # too small
    assert d(p, p, p, p, p, null, vp(512 + 16), n, 2, 8, 2, 1000, 128, 1.0, 0, null) == 3  # ws alignment
    assert d(p, p, p, p, p, vp(258), p, n, 2, 8, 2, 1000, 128, 1.0, 0, null) == 3          # lengths alignment
    assert d(p, p, p, p, p, null, p, n, 2, 8, 2, 1000, 128, 1.0, 5, null) == 1             # bad dtype
    assert lib.attn_last_launch_count() == 0


def test_dsa_argument_checks_before_any_launch(lib):
    import exact_attention_flashattention_gb300 as attn
    vp = ctypes.c_void_p
    p = vp(256)
    null = vp(0)
    f = lib.attn_dsa_bwd
    wsz = attn.attn_dsa_bwd_workspace_size
    assert wsz(1000, 576) == (1000 * 576 * 4 + 255) // 256 * 256
    assert wsz(1000, 128) == 0                # d_qk unsupported
    n = wsz(100, 576)
    # q kv o dout lse sink idx len dq dkv dsink ws bytes s_q s_kv H d_qk d_v topk scale causal stream
    ok = [p, p, p, p, p, null, p, null, p, p, null, p, n, 10, 100, 64, 576, 512, 64, 0.1, 0, null]

    def call(**kw):
        a = list(ok)
        names = ["q", "kv", "o", "dout", "lse", "sink", "idx", "len", "dq", "dkv", "dsink", "ws", "bytes",
                 "s_q", "s_kv", "H", "d_qk", "d_v", "topk", "scale", "causal", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(q=null) == 1                  # null pointer
    assert call(sink=p) == 1                  # sink without dsink
    assert call(s_q=0) == 1
    assert call(topk=0) == 1
    assert call(H=96) == 2                    # H not a multiple of 64
    assert call(d_qk=256) == 2
    assert call(d_v=256) == 2
    assert call(ws=null) == 4
    assert call(bytes=n - 1) == 4
    assert call(ws=vp(256 + 16)) == 3         # workspace alignment
    assert call(q=vp(258)) == 3               # tensor alignment
    assert call(idx=vp(258)) == 3
    assert lib.attn_last_launch_count() == 0
