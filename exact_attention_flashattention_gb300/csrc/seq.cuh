// Row addressing of the sequence dimension, shared by the forward and backward
// kernels.  A (batch, head) slice is one sequence of one head; its rows are
//   heads-major  [B, H, N, d]: row r of slice (b, h) at ((b H + h) N + r) d;
//   token-major  [tokens, H, d]: row r at ((start_b + r) H + h) d, where
//       start_b = b N (BSHD, every sequence N long) or cu[b] (packed
//       variable-length sequences, cu = B + 1 offsets, length cu[b+1] - cu[b]).
// Tiles are 128 rows of one slice.  A tile that runs past the end of its
// sequence reads rows of the next sequence (or, past the last token, the
// TMA's zero fill); the kernels mask those keys and never store those rows.
#pragma once

#include "attn_internal.h"
#include "ptx.cuh"

namespace gb300 {

struct SeqItem {
    int bh, b, h;
    int start;  // first token row of the sequence (token-major)
    int len;    // its length
};

// kTM selects the row layout at compile time: false for [B, H, N, d] (every sequence N long,
// rows of a slice contiguous), true for token-major tensors ([B, N, H, d] or packed).  The
// heads-major instantiation computes only what that layout needs.
template <bool kTM>
__device__ __forceinline__ void seq_item(const SeqDesc& s, int bh, SeqItem& it) {
    it.bh = bh;
    if constexpr (!kTM) {
        it.b = it.h = it.start = 0;  // unused by the heads-major addressing
        it.len = s.N;
        return;
    }
    it.b = bh / s.H;
    it.h = bh - it.b * s.H;
    if (s.cu != nullptr) {
        // The host never reads the offsets, so they are checked here: a sequence that does not
        // fit the token rows or the stated maximum length is skipped (no load or store touches
        // it) and reported through the error word.
        const int a = __ldg(s.cu + it.b), e = __ldg(s.cu + it.b + 1);
        if (a < 0 || e < a || e > s.tokens || e - a > s.N) {
            atomicCAS(s.error, 0, kDevBadSeqLen);
            it.start = 0;
            it.len = 0;
        } else {
            it.start = a;
            it.len = e - a;
        }
    } else {
        it.start = it.b * s.N;
        it.len = s.N;
    }
}

// TMA load of the box at column x, rows [row, row + box rows) of the slice.  The maps are
// 3-D: {d, N, B H} for heads-major tensors, {d, H, tokens} for token-major ones.
template <bool kTM>
__device__ __forceinline__ void seq_tma_load(void* dst, const CUtensorMap* map, uint64_t* bar, const SeqItem& it,
                                             int x, int row) {
    if constexpr (kTM) tma_load_3d(dst, map, bar, x, it.h, it.start + row);
    else tma_load_3d(dst, map, bar, x, row, it.bh);
}

// Element offset of (row, 0) of the slice in a [..., d] tensor.
template <bool kTM>
__device__ __forceinline__ size_t seq_row_offset(const SeqDesc& s, const SeqItem& it, int row, int d) {
    if constexpr (kTM) return ((size_t)(it.start + row) * s.H + it.h) * (size_t)d;
    else return ((size_t)it.bh * s.N + row) * (size_t)d;
}

// Index of the slice's row in L: [B, H, N] for the fixed-length layouts, [H, tokens] for
// packed sequences.
template <bool kTM>
__device__ __forceinline__ size_t seq_lse_index(const SeqDesc& s, const SeqItem& it, int row) {
    if constexpr (kTM) {
        if (s.cu != nullptr) return (size_t)it.h * s.tokens + it.start + row;
    }
    return (size_t)it.bh * s.N + row;
}

// First row of the slice in the backward's row-indexed workspace arrays, always a multiple
// of 128 (the 128-float vectors of a tile are copied with cp.async.bulk, which needs 16-byte
// aligned addresses).  Fixed length: B H blocks of n_pad = 128 ceil(N / 128) rows.  Packed:
// per head 128 (ceil(tokens / 128) + B) rows, sequence b starting at 128 (ceil(cu[b] / 128) + b).
// Consecutive sequences do not overlap: since ceil(x + y) >= ceil(x) + ceil(y) - 1, the next
// start is at least 128 ceil(len_b / 128) rows further on, the padded length of sequence b.
template <bool kTM>
__device__ __forceinline__ size_t seq_ws_base(const SeqDesc& s, const SeqItem& it, int n_pad) {
    if constexpr (kTM) {
        if (s.cu != nullptr) {
            const size_t per_head = 128 * ((size_t)(s.tokens + 127) / 128 + (size_t)s.B);
            return (size_t)it.h * per_head + 128 * ((size_t)(it.start + 127) / 128 + (size_t)it.b);
        }
    }
    return (size_t)it.bh * n_pad;
}

}  // namespace gb300
