"""Work accounting for the metric (no torch, no CUDA).

FLOP convention of "Writing Speed-of-Light Attention Backward Kernel for 5090
in CUDA" (Setup and Appendix C): the backward counts its five matmuls,
10 B H N^2 d, halved when causal (N^2/2 pairs, not N(N+1)/2); the forward
counts its two, 4 B H N^2 d, halved when causal.  Softmax, masking and scaling
are not counted.  TFLOPS = FLOPs / latency_ms / 1e9.
"""


def fwd_flops(B, H, N, d, causal):
    return 4.0 * B * H * N * N * d * (0.5 if causal else 1.0)


def bwd_flops(B, H, N, d, causal):
    return 10.0 * B * H * N * N * d * (0.5 if causal else 1.0)


def bwd_min_bytes(B, H, N, d, elem=2):
    """Lower bound on backward HBM traffic (same page, Appendix C): read Q, K, V,
    O, dO once and L (FP32) once; write dQ, dK, dV once.  Returns (read, write)."""
    bhnd = B * H * N * d
    return 5 * bhnd * elem + B * H * N * 4, 3 * bhnd * elem


def fwd_min_bytes(B, H, N, d, elem=2):
    """Read Q, K, V once; write O and L once.  Returns (read, write)."""
    bhnd = B * H * N * d
    return 3 * bhnd * elem, bhnd * elem + B * H * N * 4


def tflops(flops, ms):
    return flops / ms / 1e9
