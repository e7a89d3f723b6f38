// The backward's two HBM-bound kernels around the main kernel of attn_bwd.cu: the preprocess
// (the negated, scaled D = rowsum(dO o O), -L log2(e), and the zeroed FP32 dQ accumulator) and
// the conversion of that accumulator to 16 bits ("Writing Speed-of-Light Attention Backward
// Kernel for 5090 in CUDA", section "Mathematical Formulation": D in the dS equation; the dQ
// accumulation of the tiled backward).  They sit in their own translation unit, a module of
// their own, so that editing them leaves the main kernel's code where it is (the main kernel's
// speed was measured to move by ~1 % with its neighbours in the module).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace gb300 {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- preprocess
// ndelta_r = -scale * sum_c dO[r,c] O[r,c] (FP32: the negated D of the
// backward equations, times the softmax scale that the main kernel folds into
// dS), nlse2_r = -L_r log2(e), dq_acc[r,:] = 0.  The three workspace arrays
// hold, per (sequence, head) slice, its rows padded to whole 128-row tiles
// (seq_ws_base); the padding rows of a ragged last tile get nlse2 = -inf (so
// P = 0 there) and ndelta = 0.  Threads walk (slice, row < n_pad) with n_pad
// the padded length of the longest sequence and skip rows past a slice's own.
template <int D, bool BF16, bool kTM>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ delta,
                                                      float* __restrict__ lse2, float4* __restrict__ dq_acc,
                                                      const SeqDesc seq, int n_pad, float scale) {
    constexpr int TPR = D / 8;
    const long total = (long)seq.B * seq.H * n_pad * TPR;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const long prow = i / TPR;          // padded row of the longest sequence
        const int part = (int)(i % TPR);
        const int bh = (int)(prow / n_pad);
        const int n = (int)(prow % n_pad);
        SeqItem si;
        seq_item<kTM>(seq, bh, si);
        // the TPR threads of a row are consecutive lanes of one warp and take the same branches
        if (n >= (si.len + 127) / 128 * 128) continue;
        const size_t wrow = seq_ws_base<kTM>(seq, si, n_pad) + n;
        const bool valid = n < si.len;
        float acc = 0.f;
        if (valid) {
            const size_t src = seq_row_offset<kTM>(seq, si, n, D) / 8 + part;
            const uint4 a = __ldg(o + src);
            const uint4 b = __ldg(dout + src);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 fa, fb;
                if constexpr (BF16) {
                    fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
                    fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[e]));
                } else {
                    fa = __half22float2(*reinterpret_cast<const __half2*>(&av[e]));
                    fb = __half22float2(*reinterpret_cast<const __half2*>(&bv[e]));
                }
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
        }
        // The TPR lanes of a row (an aligned group: blocks are whole warps and total is a multiple
        // of TPR) take every branch together, so the shuffle names exactly that group.
        const unsigned lane = threadIdx.x & 31u;
        const unsigned mask = (TPR >= 32) ? 0xffffffffu : (((1u << TPR) - 1u) << (lane & ~(unsigned)(TPR - 1)));
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(mask, acc, off);
        dq_acc[2 * (wrow * TPR + part)] = make_float4(0.f, 0.f, 0.f, 0.f);
        dq_acc[2 * (wrow * TPR + part) + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (part == 0) {
            delta[wrow] = valid ? -acc * scale : 0.f;
            lse2[wrow] = valid ? -lse[seq_lse_index<kTM>(seq, si, n)] * kLog2e : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- dQ convert
// dq row n of each (sequence, head) slice = 16-bit(its accumulator row), for n below the
// sequence's length; threads walk (slice, row < N) with N the longest length.
template <int D, bool BF16, bool kTM>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq,
                                                         const SeqDesc seq, int n_pad) {
    constexpr int PER_ROW = D / 8;   // 8 values (one uint4 of output) per thread
    const long n8 = (long)seq.B * seq.H * seq.N * PER_ROW;
    const long stride = (long)gridDim.x * blockDim.x;
    if constexpr (!kTM) {
        if (seq.N == n_pad) {
            // [B, H, N, d] with whole tiles: accumulator and dq rows coincide, so the conversion is
            // a plain stream (no index arithmetic), two outputs per thread in flight.
            long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
            for (; i + stride < n8; i += 2 * stride) {
                const float4 a0 = acc[2 * i], b0 = acc[2 * i + 1];
                const float4 a1 = acc[2 * (i + stride)], b1 = acc[2 * (i + stride) + 1];
                dq[i] = make_uint4(pack2<BF16>(a0.x, a0.y), pack2<BF16>(a0.z, a0.w), pack2<BF16>(b0.x, b0.y),
                                   pack2<BF16>(b0.z, b0.w));
                dq[i + stride] = make_uint4(pack2<BF16>(a1.x, a1.y), pack2<BF16>(a1.z, a1.w),
                                            pack2<BF16>(b1.x, b1.y), pack2<BF16>(b1.z, b1.w));
            }
            if (i < n8) {
                const float4 a0 = acc[2 * i], b0 = acc[2 * i + 1];
                dq[i] = make_uint4(pack2<BF16>(a0.x, a0.y), pack2<BF16>(a0.z, a0.w), pack2<BF16>(b0.x, b0.y),
                                   pack2<BF16>(b0.z, b0.w));
            }
            return;
        }
    }
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const long row = i / PER_ROW;
        const int part = (int)(i % PER_ROW);
        const int bh = (int)(row / seq.N);
        const int n = (int)(row % seq.N);
        SeqItem si;
        seq_item<kTM>(seq, bh, si);
        if (n >= si.len) continue;
        const size_t src = ((seq_ws_base<kTM>(seq, si, n_pad) + n) * PER_ROW + part) * 2;
        const float4 a = acc[src], b = acc[src + 1];
        dq[seq_row_offset<kTM>(seq, si, n, D) / 8 + part] =
            make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w), pack2<BF16>(b.x, b.y), pack2<BF16>(b.z, b.w));
    }
}


template <int D, bool BF16, bool kTM>
cudaError_t launch_pre_t(const BwdArgs& a, cudaStream_t stream) {
    const int N_pad = (a.N + 127) / 128 * 128;
    const long threads_needed = (long)a.BH * N_pad * (D / 8);  // rows walked: every slice at the longest length
    long blocks = (threads_needed + 255) / 256;
    const long cap = (long)a.num_sms * 8;
    if (blocks > cap) blocks = cap;
    bwd_pre_kernel<D, BF16, kTM><<<(int)blocks, 256, 0, stream>>>(
        static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dout), a.lse, a.delta, a.lse2,
        reinterpret_cast<float4*>(a.dq_acc), a.seq, N_pad, a.scale);
    return cudaGetLastError();
}

template <int D, bool BF16, bool kTM>
cudaError_t launch_convert_t(const BwdArgs& a, cudaStream_t stream) {
    const int N_pad = (a.N + 127) / 128 * 128;
    const long n8 = (long)a.BH * a.N * (D / 8);
    long blocks = (n8 + 255) / 256;
    const long cap = (long)a.num_sms * 8;
    if (blocks > cap) blocks = cap;
    dq_convert_kernel<D, BF16, kTM><<<(int)blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(a.dq_acc),
                                                                static_cast<uint4*>(a.dq), a.seq, N_pad);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream) {
    const bool tm = a.seq.token_major != 0;
    if (a.d == 128) {
        if (tm) return a.fp16 ? launch_pre_t<128, false, true>(a, stream) : launch_pre_t<128, true, true>(a, stream);
        return a.fp16 ? launch_pre_t<128, false, false>(a, stream) : launch_pre_t<128, true, false>(a, stream);
    }
    if (a.d == 64) {
        if (tm) return a.fp16 ? launch_pre_t<64, false, true>(a, stream) : launch_pre_t<64, true, true>(a, stream);
        return a.fp16 ? launch_pre_t<64, false, false>(a, stream) : launch_pre_t<64, true, false>(a, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t stream) {
    const bool tm = a.seq.token_major != 0;
    if (a.d == 128) {
        if (tm) return a.fp16 ? launch_convert_t<128, false, true>(a, stream) : launch_convert_t<128, true, true>(a, stream);
        return a.fp16 ? launch_convert_t<128, false, false>(a, stream) : launch_convert_t<128, true, false>(a, stream);
    }
    if (a.d == 64) {
        if (tm) return a.fp16 ? launch_convert_t<64, false, true>(a, stream) : launch_convert_t<64, true, true>(a, stream);
        return a.fp16 ? launch_convert_t<64, false, false>(a, stream) : launch_convert_t<64, true, false>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
