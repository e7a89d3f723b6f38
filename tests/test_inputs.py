"""The seeded input generator: determinism, head independence, rounding."""
import numpy as np
import torch

import seeded_inputs as si


def test_splitmix64_published_vector():
    # SplitMix64 seeded with 1234567: first outputs of the reference generator
    # (state += 0x9E3779B97F4A7C15, then the finaliser).
    out = si.splitmix64_stream(1234567, 3)
    assert [int(x) for x in out] == [6457827717110365317, 3203168211198807973, 9817491932198370423]


def test_head_subset_matches_full_draw():
    full = si.tensor_heads(7, "q", 4, 64, 16, 1.0)
    sub = si.tensor_heads(7, "q", 4, 64, 16, 1.0, heads=[3, 1])
    assert np.array_equal(sub[0], full[3]) and np.array_equal(sub[1], full[1])
    again = si.tensor_heads(7, "q", 4, 64, 16, 1.0)
    assert np.array_equal(full, again)
    other = si.tensor_heads(7, "k", 4, 64, 16, 1.0)
    assert not np.array_equal(full, other)


def test_normal_moments():
    z = si.standard_normal(si.head_key(3, 1, 0), 1 << 18).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_bf16_rounding_matches_torch():
    x = si.standard_normal(99, 1 << 16) * np.float32(3.0)
    x = np.concatenate([x, np.array([1.00390625, 1.01171875, -2.0, 0.0], np.float32)])  # ties
    ours = si.round_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = si.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_fp16_rounding_matches_torch():
    x = si.standard_normal(98, 1 << 16)
    ours = si.round_fp16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_late_spike_puts_max_in_last_tile():
    N, d = 256, 16
    q = si.tensor_heads(5, "q", 1, N, d, 1.0)[0]
    k = si.tensor_heads(5, "k", 1, N, d, 1.0)[0]
    rows = [130, 200, 255]
    k2 = si.late_spike(q, k, "bf16", 40.0, rows)
    qf, kf = si.bits_to_f32(q, "bf16"), si.bits_to_f32(k2, "bf16")
    for i in rows:
        s = kf[: i + 1] @ qf[i]
        assert s.argmax() >= 128
