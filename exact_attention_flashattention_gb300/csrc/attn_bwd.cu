// Fused attention backward for sm_103a: the main tcgen05 kernel, launched between
// the preprocess and the dQ conversion of bwd_aux.cu ("Writing Speed-of-Light Attention Backward Kernel for 5090
// in CUDA", sections "Mathematical Formulation" and the tiled pseudocode that
// follows it: one CTA owns dK_j and dV_j of a key/value tile j, loops over the
// query tiles i it interacts with, and adds each dQ_i partial into an FP32
// accumulator; a second kernel converts that accumulator after a kernel
// boundary).
//
// sm_103a mapping (transposed formulation, keys on TMEM lanes):
//   S^T  = K_j Q_i^T      SS-MMA  -> TMEM [256,384)   (P^T written over it)
//   dP^T = V_j dO_i^T     SS-MMA  -> TMEM [384,512)   (dS^T written over it)
//   dV  += P^T dO_i       TS-MMA  (A = P^T from TMEM) -> TMEM [0,128)
//   dK  += dS^T Q_i       TS-MMA  (A = dS^T from TMEM) -> TMEM [128,256)
//   dQ_i^T = K_j^T dS^T   SS-MMA  (d = 128; dS^T from shared memory) -> TMEM [384,512)
//   dQ_i   = dS K_j       SS-MMA  (d = 64, same operands swapped)      -> TMEM [384,448)
// dS is stored already multiplied by the softmax scale, so dK and the dQ
// partials need no further scaling.  With d = 128 the dQ partial comes out
// transposed (head dimension on the TMEM lanes): a warp's FP32 reductions into
// the accumulator then cover 32 consecutive floats of one row (a full 128-byte
// line) instead of 16 bytes of 32 different rows.
// The transposes follow from the equations: dV = P^T dO and dK = dS^T Q need
// P^T and dS^T as the left operand, which the tensor core can read straight
// from TMEM when the scores are computed with keys on the lanes.
//
// CTA layout (512 threads): warps 0-7 elementwise (P, dS; warp w handles TMEM
// lane quadrant w%4 and query columns [64 (w/4), +64)), warps 8-11 dQ drain
// and dK/dV epilogue, warp 12 MMA issuer (owns TMEM), warp 13 TMA producer, warp 15
// (packed sequences) the thread that takes units from the work counter.
#include "attn_internal.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace gb300 {
namespace {

constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPanelBytes = 128 * 128;
// SM cycles over which a dQ drain spreads one tile's accumulator reductions (the window also
// bounds how late the drain can start the next tile).  Measured, backward of causal B=8 H=16
// N=4096 d=128: 1500 / 2000 / 2500 / 2750 / 3000 / 3250 / 3500 / 4000 cycles gave 1.28 / 1.28 /
// 1.26 / 1.23 / 1.22 / 1.24 / 1.29 / 1.30 ms against 1.38 ms unpaced; causal B=4 H=16 N=4096
// d=64: 1500 / 2500 / 3000 / 3500 gave 0.586 / 0.562 / 0.518 / 0.516 ms against 0.592.
template <int D>
constexpr long long kDqPaceCycles = D == 128 ? 3000 : 3500;

// ---------------------------------------------------------------- main kernel
// Shared memory: K_j, V_j (one tile each), Q_i and dO_i (two stages each), dS
// (128 x 128 16-bit, written by the elementwise warps as the MN-major A operand
// of dQ = dS K_j), and per stage the 128 values of -L log2(e) and of -D.
template <int D>
struct BwdLayout {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kQ = 2 * kTile;          // [2 stages]
    static constexpr int kDO = 4 * kTile;         // [2 stages]
    static constexpr int kDS = 6 * kTile;         // 2 panels of 128 rows x 128 bytes
    static constexpr int kVec = kDS + 2 * kPanelBytes;  // [2 stages][-L log2 e (128) | -D (128)] FP32
    static constexpr int kAux = kVec + 2 * 256 * 4;
    static constexpr int kBarKFull = 0, kBarKEmpty = 1, kBarVFull = 2, kBarVEmpty = 3;
    static constexpr int kBarQFull = 4;    // [2]: Q_i, dO_i and the two vectors of stage i % 2
    static constexpr int kBarQEmpty = 6;   // [2]
    static constexpr int kBarSFull = 8, kBarDpFull = 9, kBarPReady = 10, kBarDsReady = 11;
    static constexpr int kBarDqFull = 12, kBarDqFree = 13, kBarDkvFull = 14, kBarDkvEmpty = 15;
    static constexpr int kBarTeardown = 16;
    static constexpr int kBarSchedFull = 17;    // [4] packed sequences: dynamic unit distribution
    static constexpr int kBarSchedEmpty = 21;   // [4]
    static constexpr int kNumBars = 25;
    static constexpr int kSchedSlotWord = 2 * kNumBars;  // int index of the ring's 4 unit slots
    static constexpr int kMiscOff = kAux + kNumBars * 8 + 16;
    static constexpr int kBytes = kMiscOff + 16;
    // TMEM columns: dV, dK accumulators; S^T (P^T packed over it); dP^T (dS^T packed over it),
    // reused for the dQ_i tile once dK has consumed dS^T.
    static constexpr int kTmemDV = 0, kTmemDK = 128, kTmemS = 256, kTmemDP = 384, kTmemDQ = 384;
};

struct BwdItem {
    SeqItem si;         // the (sequence, head) slice
    int T;              // its number of 128-row tiles
    int j, i0, n;       // key/value tile, first query tile, number of query tiles
};

// Work list.  Causal: units of two key/value tiles of one head, j and T-1-j, longest first.
// Tile j meets T-j query tiles, so every unit holds T+1 of them and a static round-robin of
// units over the persistent CTAs is balanced.  Non-causal: one tile per unit (all equally
// long; a finer grain shortens the tail).  Consecutive units share a head, so the CTAs
// running at one time reuse that head's Q / dO from L2.  Units are laid out for the longest
// sequence (T tiles); a shorter packed sequence skips the units past its own tiles (slot 0
// is skipped only when slot 1 is too, so the callers stop at the first skipped slot).
__device__ __forceinline__ int bwd_units_per_head(int T, int causal) { return causal ? (T + 1) / 2 : T; }

template <bool kTM>
__device__ __forceinline__ bool bwd_item(int u, int s, int T, int causal, const SeqDesc& seq, BwdItem& w) {
    const int uph = bwd_units_per_head(T, causal);
    const int jp = u % uph;
    seq_item<kTM>(seq, u / uph, w.si);
    w.T = (w.si.len + 127) / 128;
    if (causal) {
        const int jl = w.T - 1 - jp;
        if (jl < jp) return false;
        if (s == 1 && jl == jp) return false;
        w.j = s ? jl : jp;
    } else {
        if (s == 1 || jp >= w.T) return false;
        w.j = jp;
    }
    w.i0 = causal ? w.j : 0;
    w.n = w.T - w.i0;
    return true;
}

// Dynamic distribution for packed sequences of different lengths, as in the forward: one
// thread takes units from the launch's counter and publishes them through a 4-entry ring in
// the barrier area; every role reads the same sequence of units, holds an entry until its unit
// is done, releases it with its own arrival, and the scheduler claims at most one unit ahead.
// Consumers: the 256 elementwise threads, the 128 drain threads, the MMA warp and the TMA
// thread.
constexpr int kSchedDepth = 4;
constexpr int kSchedAhead = 1;
constexpr int kBwdSchedConsumers = 256 + 128 + 32 + 1;

// This CTA's sequence of units; next() returns the next unit, or -1 at the end (or when a
// wait gave up).  kDyn = false: blockIdx.x, blockIdx.x + gridDim.x, ...
template <bool kDyn>
struct BwdUnits;

template <>
struct BwdUnits<false> {
    int u;
    const int n_units;
    __device__ explicit BwdUnits(int n) : u((int)blockIdx.x - (int)gridDim.x), n_units(n) {}
    template <class L>
    __device__ int next(uint64_t*, const WaitGuard&, int) {
        u += (int)gridDim.x;
        return u < n_units ? u : -1;
    }
};

template <>
struct BwdUnits<true> {
    uint32_t k = 0;   // ring entries taken
    __device__ explicit BwdUnits(int) {}
    template <class L>
    __device__ int next(uint64_t* bars, const WaitGuard& g, int code) {
        const volatile int* ring = reinterpret_cast<volatile int*>(bars) + L::kSchedSlotWord;
        if (k > 0) mbar_arrive(&bars[L::kBarSchedEmpty + (k - 1) % kSchedDepth]);
        if (!mbar_wait(&bars[L::kBarSchedFull + k % kSchedDepth], (k / kSchedDepth) & 1, g, code)) return -1;
        return ring[k++ % kSchedDepth];
    }
};

template <int D, bool BF16, bool kTM, bool kDyn>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const float* __restrict__ nlse2, const float* __restrict__ ndelta, float* __restrict__ dq_acc,
                void* __restrict__ dk_out, void* __restrict__ dv_out, const SeqDesc seq, float scale, int causal,
                int smem_slack, unsigned int* __restrict__ sched, int* error) {
    using L = BwdLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if ((int)pad > smem_slack) {
        // The tiles need 1024-byte alignment and the launch could not give this much slack.
        if (threadIdx.x == 0) atomicCAS(error, 0, kDevSmemAlign);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kAux);
    const float* vec = reinterpret_cast<const float*>(smem + L::kVec);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = (seq.N + 127) / 128;  // tiles of the longest sequence (the last one may be ragged)
    const int N_pad = T * 128;          // rows per slice of the fixed-length workspace arrays
    const int n_units = seq.B * seq.H * bwd_units_per_head(T, causal);

    if (threadIdx.x == 0) {
        for (int b = 0; b < L::kBarSchedFull; ++b) mbar_init(&bars[b], 1);
        if (kDyn) {
            for (int b = 0; b < kSchedDepth; ++b) {
                mbar_init(&bars[L::kBarSchedFull + b], 1);
                mbar_init(&bars[L::kBarSchedEmpty + b], kBwdSchedConsumers);
            }
        }
        mbar_init(&bars[L::kBarPReady], 256);
        mbar_init(&bars[L::kBarDsReady], 256);
        mbar_init(&bars[L::kBarDqFree], 128);
        mbar_init(&bars[L::kBarDkvEmpty], 128);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 12) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 13 && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard guard{abort_flag, error, kWaitLimitNs};
    const float scale_log2 = scale * kLog2e;

    if (warp < 8) {
        // ------------------------------------------------------ P and dS (elementwise)
        regs_inc<144>();
        const int half = warp >> 2;              // query columns [64 half, 64 half + 64)
        const int row = (warp & 3) * 32 + lane;  // key row within the tile (TMEM lane)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + L::kTmemS + 64 * half;
        const uint32_t dp_addr = tmem + lane_base + L::kTmemDP + 64 * half;
        uint8_t* ds_panel = smem + L::kDS + half * kPanelBytes;
        const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
        const uint64_t sc2 = f2_pack(scale, scale);
        uint32_t g = 0;
        bool ok = true;
        BwdUnits<kDyn> units(n_units);
        for (int u; ok && (u = units.template next<L>(bars, guard, kDevTimeoutSoftmax)) >= 0;) {
            for (int sidx = 0; sidx < 2 && ok; ++sidx) {
                BwdItem w;
                if (!bwd_item<kTM>(u, sidx, T, causal, seq, w)) break;
                for (int it = 0; it < w.n; ++it, ++g) {
                    const int i = w.i0 + it;
                    const bool diag = causal && i == w.j;
                    const float2* nl = reinterpret_cast<const float2*>(vec + (g & 1) * 256 + 64 * half);
                    const float2* nd = reinterpret_cast<const float2*>(vec + (g & 1) * 256 + 128 + 64 * half);
                    // P^T = 2^(S^T scale log2 e - L log2 e), keys > queries masked on the diagonal tile
                    if (!mbar_wait(&bars[L::kBarSFull], g & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                    tc_fence_after();
                    float p[64];
                    {
                        uint32_t s[64];
                        tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                        tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float2 l = nl[e];
                            const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])),
                                                      sl2, f2_pack(l.x, l.y));
                            float x0, x1;
                            f2_unpack(x, x0, x1);
                            p[2 * e] = ex2_ftz(x0);
                            p[2 * e + 1] = ex2_ftz(x1);
                        }
                        if (diag) {
#pragma unroll
                            for (int e = 0; e < 64; ++e)
                                if (row > 64 * half + e) p[e] = 0.f;
                        }
                        if (w.j * 128 + row >= w.si.len) {
                            // a key past the end of the sequence in its ragged last tile
#pragma unroll
                            for (int e = 0; e < 64; ++e) p[e] = 0.f;
                        }
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(p[32 * c + 2 * e], p[32 * c + 2 * e + 1]);
                            tmem_st16(s_addr + 16 * c, pk);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars[L::kBarPReady]);

                    // scale dS^T = P^T o (scale dP^T - scale D): into TMEM (A operand of dK) and shared
                    // memory (an operand of the dQ product)
                    if (!mbar_wait(&bars[L::kBarDpFull], g & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                    if (!mbar_wait(&bars[L::kBarDqFull], (g & 1) ^ 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t dp[32];
                        tmem_ld32(dp_addr + 32 * c, dp);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 dl = nd[16 * c + e];
                            const uint64_t t = f2_fma(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                                      sc2, f2_pack(dl.x, dl.y));
                            const uint64_t ds = f2_mul(f2_pack(p[32 * c + 2 * e], p[32 * c + 2 * e + 1]), t);
                            float d0, d1;
                            f2_unpack(ds, d0, d1);
                            pk[e] = pack2<BF16>(d0, d1);
                        }
                        tmem_st16(dp_addr + 16 * c, pk);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint4* dst = reinterpret_cast<uint4*>(ds_panel + sw128_offset(row, 4 * c + e));
                            *dst = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars[L::kBarDsReady]);
                }
            }
        }
    } else if (warp < 12) {
        // ------------------------------------------------------ dQ drain, dK/dV epilogue
        // d = 128 holds a whole 128-column dQ^T tile in registers; d = 64 needs fewer.
        if constexpr (D == 128) regs_inc<136>(); else regs_dec<112>();
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t g = 0;
        int k = 0;
        bool ok = true;
        const bool kv_al32 = ((reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) & 31u) == 0;
        BwdUnits<kDyn> units(n_units);
        for (int u; ok && (u = units.template next<L>(bars, guard, kDevTimeoutCorr)) >= 0;) {
            for (int sidx = 0; sidx < 2 && ok; ++sidx, ++k) {
                BwdItem w;
                if (!bwd_item<kTM>(u, sidx, T, causal, seq, w)) break;
                for (int it = 0; it < w.n; ++it, ++g) {
                    const int i = w.i0 + it;
                    if (!mbar_wait(&bars[L::kBarDqFull], g & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                    tc_fence_after();
                    if constexpr (D == 128) {
                        // dQ_i^T: this thread holds column `row` (a head-dimension index) of dQ_i for
                        // all 128 query rows; one warp instruction covers 32 consecutive floats of a
                        // row.  The whole tile is read out of TMEM (and its columns released to the
                        // next dP^T) before the reductions are issued.
                        float* dst = dq_acc + (seq_ws_base<kTM>(seq, w.si, N_pad) + (size_t)i * 128) * D + row;
                        uint32_t r[128];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            tmem_ld32(tmem + lane_base + L::kTmemDQ + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
                        tmem_wait_ld();
                        tc_fence_before();
                        mbar_arrive(&bars[L::kBarDqFree]);
                        // The tile's 128 reductions are spread over kDqPaceCycles (four every
                        // kDqPaceCycles / 32 cycles) instead of going out back to back.  Every CTA
                        // adds 64 KB per query tile, and in one burst these queue at L2 ahead of the
                        // next Q_i / dO_i loads, which then take about twice as long to land and stall
                        // the MMA issuer.  The wait is a spin on the SM clock and ends by itself.
                        const long long t0 = clock64();
#pragma unroll
                        for (int e = 0; e < 128; ++e) {
                            red_add_f32(dst + (size_t)e * D, __uint_as_float(r[e]));
                            if ((e & 3) == 3 && e < 127) {
                                const long long due = t0 + (long long)(e + 1) * kDqPaceCycles<D> / 128;
                                while (clock64() < due) {}
                            }
                        }
                    } else {
                        // dQ_i: this thread holds query row `row`.
                        float* dst = dq_acc + (seq_ws_base<kTM>(seq, w.si, N_pad) + (size_t)i * 128 + row) * D;
                        uint32_t r[64];
                        tmem_ld32(tmem + lane_base + L::kTmemDQ, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                        tmem_ld32(tmem + lane_base + L::kTmemDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                        tmem_wait_ld();
                        tc_fence_before();
                        mbar_arrive(&bars[L::kBarDqFree]);
                        // paced as at d = 128: one 16-byte reduction every kDqPaceCycles / 16 cycles
                        const long long t0 = clock64();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            red_add_v4(dst + 4 * e, __uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                       __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
                            if (e < 15) {
                                const long long due = t0 + (long long)(e + 1) * kDqPaceCycles<D> / 16;
                                while (clock64() < due) {}
                            }
                        }
                    }
                }
                if (!ok) break;
                if (!mbar_wait(&bars[L::kBarDkvFull], k & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                tc_fence_after();
                const bool row_valid = w.j * 128 + row < w.si.len;
                const size_t grow_off = seq_row_offset<kTM>(seq, w.si, w.j * 128 + row, D);
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint32_t src = tmem + lane_base + (which ? L::kTmemDK : L::kTmemDV);
                    uint8_t* dst = reinterpret_cast<uint8_t*>(which ? dk_out : dv_out) + grow_off * 2;
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(src + c, r);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack2<BF16>(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                        if (row_valid) {
                            // one row per thread: 32-byte stores fill whole sectors (rows start at
                            // multiples of 128 bytes, so a 32-byte aligned base suffices)
                            if (kv_al32) {
                                st_global_v8(dst + c * 2, &pk[0]);
                                st_global_v8(dst + c * 2 + 32, &pk[8]);
                            } else {
                                uint4* d4 = reinterpret_cast<uint4*>(dst + c * 2);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[L::kBarDkvEmpty]);
            }
        }
    } else {
        // warps 12-15; the split 2 x 144 + 136 + 88 (d = 128) or 2 x 144 + 112 + 112 (d = 64)
        // uses exactly the 65536 registers the block is launched with
        if constexpr (D == 128) regs_dec<88>(); else regs_dec<112>();
        if (warp == 12) {
            // ------------------------------------------------------ MMA issuer (the whole warp; lane 0 issues)
            constexpr uint32_t kIdescS = idesc_f16(128, 128, BF16, false, false);   // S^T, dP^T
            constexpr uint32_t kIdescG = idesc_f16(128, D, BF16, false, true);      // dV, dK (A in TMEM)
            constexpr uint32_t kIdescQ = idesc_f16(128, D == 128 ? 128 : D, BF16, true, true);  // dQ^T or dQ
            const uint32_t k_base = smem_u32(smem + L::kK), v_base = smem_u32(smem + L::kV);
            const uint32_t q_base = smem_u32(smem + L::kQ), do_base = smem_u32(smem + L::kDO);
            const uint32_t ds_base = smem_u32(smem + L::kDS);
            uint32_t g = 0;
            int k = 0;
            bool ok = true;
            constexpr bool kDqAfterS = (D == 64);
            // d = 128: dQ_i^T = K_j^T dS^T (A = K_j read MN-major, B = dS^T MN-major).
            // d = 64:  dQ_i = dS K_j (A = dS^T read MN-major, B = K_j MN-major).
            // Reads the dS tile in shared memory; writes the dP^T columns (dK has read dS^T there).
            const uint64_t kd_mn = sdesc_sw128(k_base, kPanelBytes, 1024);
            const uint64_t sd_mn = sdesc_sw128(ds_base, kPanelBytes, 1024);
            auto issue_dq = [&]() {
                if constexpr (D == 128)
                    warp_mma_ss8<GB300_MNMAJ_OFFS, GB300_MNMAJ_OFFS>(tmem + L::kTmemDQ, kd_mn, sd_mn, kIdescQ, 0);
                else
                    warp_mma_ss8<GB300_MNMAJ_OFFS, GB300_MNMAJ_OFFS>(tmem + L::kTmemDQ, sd_mn, kd_mn, kIdescQ, 0);
                warp_mma_commit(&bars[L::kBarDqFull]);
            };
            // S^T = K_j Q_i^T and dP^T = V_j dO_i^T: K-major operands, D / 16 steps
            auto issue_kmajor = [&](uint32_t d_col, uint32_t a_base, uint32_t b_base) {
                const uint64_t ad = sdesc_sw128(a_base, 16, 1024), bd = sdesc_sw128(b_base, 16, 1024);
                if constexpr (D == 128)
                    warp_mma_ss8<GB300_KMAJ_OFFS(kPanelBytes), GB300_KMAJ_OFFS(kPanelBytes)>(tmem + d_col, ad, bd,
                                                                                          kIdescS, 0);
                else
                    warp_mma_ss4<2, 4, 6, 2, 4, 6>(tmem + d_col, ad, bd, kIdescS, 0);
            };
            BwdUnits<kDyn> units(n_units);
            for (int u; ok && (u = units.template next<L>(bars, guard, kDevTimeoutMma)) >= 0;) {
                for (int sidx = 0; sidx < 2 && ok; ++sidx, ++k) {
                    BwdItem w;
                    if (!bwd_item<kTM>(u, sidx, T, causal, seq, w)) break;
                    if (!warp_mbar_wait(&bars[L::kBarKFull], k & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                    if (!warp_mbar_wait(&bars[L::kBarVFull], k & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                    tc_fence_after();
                    // S^T = K_j Q_i^T into the S columns (last read by the previous dV, issued earlier)
                    auto issue_s = [&](uint32_t gg) -> bool {
                        const uint32_t sst = gg & 1;
                        if (!warp_mbar_wait(&bars[L::kBarQFull + sst], (gg >> 1) & 1, guard, kDevTimeoutMma)) return false;
                        tc_fence_after();
                        issue_kmajor(L::kTmemS, k_base, q_base + sst * L::kTile);
                        warp_mma_commit(&bars[L::kBarSFull]);
                        return true;
                    };
                    for (int it = 0; it < w.n; ++it, ++g) {
                        const uint32_t st = g & 1;
                        const uint32_t qs = q_base + st * L::kTile, dos = do_base + st * L::kTile;
                        // d = 128: S^T of query tile i was issued after dV of tile i - 1 (below), so
                        // the elementwise warps can start its P^T while dK and dQ^T of i - 1 run.
                        if (kDqAfterS || it == 0) {
                            if (!issue_s(g)) { ok = false; break; }
                        } else {
                            if (!warp_mbar_wait(&bars[L::kBarQFull + st], (g >> 1) & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                            tc_fence_after();
                        }
                        // d = 64: the previous query tile's dQ goes between S^T and dP^T, so the
                        // elementwise P^T pass overlaps it as well as dP^T.  d = 128: it stays at the
                        // end of the previous tile, where S^T hides the longer drain of its reductions
                        // (measured: 949 vs 877 TFLOPS at d = 128; 505 vs 532 at d = 64).
                        if (kDqAfterS && it > 0) issue_dq();
                        // dP^T = V_j dO_i^T, once the previous dQ tile has left these columns
                        if (!warp_mbar_wait(&bars[L::kBarDqFree], (g & 1) ^ 1, guard, kDevTimeoutMma)) { ok = false; break; }
                        tc_fence_after();
                        issue_kmajor(L::kTmemDP, v_base, dos);
                        warp_mma_commit(&bars[L::kBarDpFull]);
                        if (it == w.n - 1) warp_mma_commit(&bars[L::kBarVEmpty]);
                        // dV += P^T dO_i
                        if (!warp_mbar_wait(&bars[L::kBarPReady], g & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                        if (it == 0 && !warp_mbar_wait(&bars[L::kBarDkvEmpty], (k & 1) ^ 1, guard, kDevTimeoutMma)) { ok = false; break; }
                        tc_fence_after();
                        warp_mma_ts8<GB300_TMEM_A_OFFS, GB300_MNMAJ_OFFS>(
                            tmem + L::kTmemDV, tmem + L::kTmemS, sdesc_sw128(dos, kPanelBytes, 1024), kIdescG, it > 0);
                        if (!kDqAfterS && it + 1 < w.n && !issue_s(g + 1)) { ok = false; break; }
                        // dK += dS^T Q_i
                        if (!warp_mbar_wait(&bars[L::kBarDsReady], g & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                        tc_fence_after();
                        warp_mma_ts8<GB300_TMEM_A_OFFS, GB300_MNMAJ_OFFS>(
                            tmem + L::kTmemDK, tmem + L::kTmemDP, sdesc_sw128(qs, kPanelBytes, 1024), kIdescG, it > 0);
                        warp_mma_commit(&bars[L::kBarQEmpty + st]);
                        if (!kDqAfterS) issue_dq();
                    }
                    if (!ok) break;
                    if (kDqAfterS) issue_dq();  // the item's last dQ tile
                    warp_mma_commit(&bars[L::kBarKEmpty]);
                    warp_mma_commit(&bars[L::kBarDkvFull]);
                }
            }
            warp_mma_commit(&bars[L::kBarTeardown]);
            mbar_wait_drain(&bars[L::kBarTeardown], 0, kWaitLimitNs);
        } else if (kDyn && warp == 15 && lane == 0) {
            // ------------------------------------------------------ scheduler (packed sequences)
            for (uint32_t k = 0;; ++k) {
                const uint32_t pos = k % kSchedDepth, e = k - 1 - kSchedAhead;  // e: entry to be released
                if (k > (uint32_t)kSchedAhead &&
                    !mbar_wait_sleep(&bars[L::kBarSchedEmpty + e % kSchedDepth], (e / kSchedDepth) & 1, guard,
                                     kDevTimeoutLoad))
                    break;
                const unsigned int u = atomicAdd(sched, 1u);
                const int val = u < (unsigned int)n_units ? (int)u : -1;
                reinterpret_cast<volatile int*>(bars)[L::kSchedSlotWord + pos] = val;
                mbar_arrive(&bars[L::kBarSchedFull + pos]);  // release: the slot is written first
                if (val < 0) break;
            }
        } else if (warp == 13 && lane == 0) {
            // ------------------------------------------------------ TMA producer
            uint32_t g = 0;
            int k = 0;
            bool ok = true;
            int last_kv = -1;
            auto load_q = [&](const BwdItem& w, int it) -> bool {
                const int i = w.i0 + it;
                const uint32_t st = g & 1;
                if (!mbar_wait(&bars[L::kBarQEmpty + st], ((g >> 1) & 1) ^ 1, guard, kDevTimeoutLoad)) return false;
                mbar_arrive_expect_tx(&bars[L::kBarQFull + st], 2 * L::kTile + 1024);
#pragma unroll
                for (int p = 0; p < L::kPanels; ++p) {
                    seq_tma_load<kTM>(smem + L::kQ + st * L::kTile + p * kPanelBytes, &tm_q, &bars[L::kBarQFull + st],
                                 w.si, 64 * p, i * 128);
                    seq_tma_load<kTM>(smem + L::kDO + st * L::kTile + p * kPanelBytes, &tm_do, &bars[L::kBarQFull + st],
                                 w.si, 64 * p, i * 128);
                }
                const size_t r0 = seq_ws_base<kTM>(seq, w.si, N_pad) + (size_t)i * 128;
                bulk_load(smem + L::kVec + st * 1024, nlse2 + r0, 512, &bars[L::kBarQFull + st]);
                bulk_load(smem + L::kVec + st * 1024 + 512, ndelta + r0, 512, &bars[L::kBarQFull + st]);
                ++g;
                return true;
            };
            BwdUnits<kDyn> units(n_units);
            for (int u; ok && (u = units.template next<L>(bars, guard, kDevTimeoutLoad)) >= 0;) {
                for (int sidx = 0; sidx < 2 && ok; ++sidx, ++k) {
                    BwdItem w;
                    if (!bwd_item<kTM>(u, sidx, T, causal, seq, w)) break;
                    // V_j as soon as the previous item's last dP^T is done, then the first Q_i / dO_i,
                    // then K_j once the previous item's last dQ is done, then the rest.
                    if (!mbar_wait(&bars[L::kBarVEmpty], (k & 1) ^ 1, guard, kDevTimeoutLoad)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars[L::kBarVFull], L::kTile);
#pragma unroll
                    for (int p = 0; p < L::kPanels; ++p)
                        seq_tma_load<kTM>(smem + L::kV + p * kPanelBytes, &tm_v, &bars[L::kBarVFull], w.si, 64 * p, w.j * 128);
                    if (!load_q(w, 0)) { ok = false; break; }
                    if (!mbar_wait(&bars[L::kBarKEmpty], (k & 1) ^ 1, guard, kDevTimeoutLoad)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars[L::kBarKFull], L::kTile);
                    last_kv = k;
#pragma unroll
                    for (int p = 0; p < L::kPanels; ++p)
                        seq_tma_load<kTM>(smem + L::kK + p * kPanelBytes, &tm_k, &bars[L::kBarKFull], w.si, 64 * p, w.j * 128);
                    for (int it = 1; it < w.n && ok; ++it)
                        if (!load_q(w, it)) ok = false;
                }
            }
            // Let every copy issued above land before shared memory is released.
            if (last_kv >= 0) {
                mbar_wait_drain(&bars[L::kBarKFull], last_kv & 1, kWaitLimitNs);
                mbar_wait_drain(&bars[L::kBarVFull], last_kv & 1, kWaitLimitNs);
            }
            for (uint32_t t = (g > 2 ? g - 2 : 0); t < g; ++t)
                mbar_wait_drain(&bars[L::kBarQFull + (t & 1)], (t >> 1) & 1, kWaitLimitNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool BF16, bool kTM>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream, int stage) {
    using L = BwdLayout<D>;
    const int T = (a.N + 127) / 128;
    // 1. preprocess (bwd_aux.cu)
    if (stage < 0 || stage == 0) {
        cudaError_t e = launch_bwd_pre(a, stream);
        if (e != cudaSuccess) return e;
    }
    // 2. main kernel
    if (stage < 0 || stage == 1) {
        int max_smem = 0;
        cudaError_t e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, a.device);
        if (e != cudaSuccess) return e;
        const int want = L::kBytes + 1024;
        const int smem_bytes = want < max_smem ? want : max_smem;
        const int slack = smem_bytes - L::kBytes;
        if (slack < 0) return cudaErrorInvalidConfiguration;
        // Packed sequences of different lengths take units from the launch's counter; the
        // fixed-length layouts keep the static split (their units all carry the same work).
        auto kern = attn_bwd_kernel<D, BF16, kTM, false>;
        if constexpr (kTM) {
            if (a.seq.cu != nullptr) kern = attn_bwd_kernel<D, BF16, kTM, true>;
        }
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        const long n_units = (long)a.BH * (a.causal ? (T + 1) / 2 : T);
        const int grid = (int)(n_units < a.num_sms ? n_units : a.num_sms);
        kern<<<grid, kThreads, smem_bytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse2, a.delta, a.dq_acc,
                                                      a.dk, a.dv, a.seq, a.scale, a.causal, slack, a.sched, a.error);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // 3. dQ conversion (bwd_aux.cu)
    if (stage < 0 || stage == 2) {
        cudaError_t e = launch_dq_convert(a, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <bool kTM>
cudaError_t launch_bwd_l(const BwdArgs& a, cudaStream_t stream, int stage) {
    if (a.d == 128)
        return a.fp16 ? launch_bwd_t<128, false, kTM>(a, stream, stage) : launch_bwd_t<128, true, kTM>(a, stream, stage);
    if (a.d == 64)
        return a.fp16 ? launch_bwd_t<64, false, kTM>(a, stream, stage) : launch_bwd_t<64, true, kTM>(a, stream, stage);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stage) {
    return a.seq.token_major ? launch_bwd_l<true>(a, stream, stage) : launch_bwd_l<false>(a, stream, stage);
}

}  // namespace gb300
