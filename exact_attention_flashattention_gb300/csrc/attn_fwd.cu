// Fused attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// Computes, per (batch, head), S = scale * Q K^T + M, the row log-sum-exp L,
// P = exp(S - L) and O = P V without writing S or P to global memory
// ("Writing Speed-of-Light Attention Backward Kernel for 5090 in CUDA",
// section "Mathematical Formulation", forward equations).  The running-max
// (online) softmax follows "Dense B200 attention from scratch" (b200-attention),
// Chapter 1 section B; the kernel organisation (warp roles, two Q tiles per
// CTA, a K/V ring, the peeled compute pipeline, base-2 exponentials with the
// scale folded in, the lazy O rescale with threshold 8 and the separate
// correction warps, persistent CTAs) follows its Chapters 4-8, 11, 12 and 14,
// re-derived for sm_103a.  Causal tile skipping is added; that page's kernel
// is non-causal.
//
// CTA layout (512 threads = 4 warpgroups):
//   WG0 (warps 0-3)   softmax for Q tile 0 of the work item (row = thread)
//   WG1 (warps 4-7)   softmax for Q tile 1
//   WG2 (warps 8-11)  O correction (lazy rescale) and the epilogue
//   WG3 warp 12       tcgen05.mma issuer: the whole warp waits, one lane issues (also owns TMEM)
//   WG3 warp 13       TMA producer, K/V ring
//   WG3 warp 14       TMA producer, Q tiles
//   WG3 warp 15       idle (packed sequences: lane 0 takes units from the work counter)
// TMEM (512 columns x 128 lanes): S0 [0,128) S1 [128,256) O0 [256,..) O1 [384,..).
// Packed 16-bit P_q overwrites the first 64 columns of S_q.
// Shared memory: Q0, Q1 (128 x d each) and a ring of K/V tiles (128 x d),
// all in the 128-byte-swizzle layout written by TMA.
#include "attn_internal.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace gb300 {
namespace {

constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // base-2 units (b200-attention, Chapter 11)
constexpr int kPanelBytes = 128 * 128;     // 128 rows x 128 bytes (64 16-bit elements)

// Dynamic work distribution: one thread of the CTA takes units from a global counter (so a CTA
// that finishes early takes more, which balances units of unequal work, e.g. packed sequences
// of different lengths) and publishes them, in order, through a ring in shared memory; -1 ends
// the sequence.  Every role reads the same sequence and expands each unit into its items.  Each
// entry is held until its unit is done, and the scheduler claims entry k only once every
// consumer has released entry k - 1 - kSchedAhead, so a CTA holds at most kSchedAhead units
// beyond the one it works on: enough to hide the atomic's latency, little to hold back at the
// end of the work.
constexpr int kSchedDepth = 4;
constexpr int kSchedAhead = 1;
static_assert(kSchedAhead + 1 <= kSchedDepth, "a slot is rewritten only after its entry was released");

template <int D>
struct FwdLayout {
    static constexpr int kTile = 128 * D * 2;          // bytes of a 128-row tile
    static constexpr int kPanels = D / 64;
    static constexpr int kStages = (D == 128) ? 4 : 6;  // K/V ring depth
    static constexpr int kQ0 = 0;
    static constexpr int kQ1 = kTile;
    static constexpr int kKV = 2 * kTile;
    static constexpr int kAux = kKV + kStages * kTile;  // barriers and small arrays
    // aux area
    static constexpr int kBarQFull = 0, kBarQEmpty = 1;
    static constexpr int kBarKVFull = 2;
    static constexpr int kBarKVEmpty = kBarKVFull + kStages;
    static constexpr int kBarSFull = kBarKVEmpty + kStages;  // [2]
    static constexpr int kBarPVReady = kBarSFull + 2;        // [2]
    static constexpr int kBarODone = kBarPVReady + 2;        // [2]
    static constexpr int kBarStats = kBarODone + 2;          // [2]
    static constexpr int kBarFin = kBarStats + 2;            // [2 stages][2 buffers]
    static constexpr int kBarTeardown = kBarFin + 4;
    static constexpr int kBarSchedFull = kBarTeardown + 1;  // [kSchedDepth]
    static constexpr int kBarSchedEmpty = kBarSchedFull + kSchedDepth;  // [kSchedDepth]
    static constexpr int kNumBars = kBarSchedEmpty + kSchedDepth;
    static constexpr int kSchedSlotWord = 2 * kNumBars;  // int index of the ring's 4 unit slots, after the barriers
    static constexpr int kScaleOff = kAux + 8 * 64;                // float [2][128]
    static constexpr int kFinLOff = kScaleOff + 2 * 128 * 4;       // float [2 buf][2 q][128]
    static constexpr int kFinMOff = kFinLOff + 4 * 128 * 4;        // float [2 buf][2 q][128]
    static constexpr int kMiscOff = kFinMOff + 4 * 128 * 4;        // tmem base, abort flag
    static constexpr int kBytes = kMiscOff + 64;
    static constexpr int kTmemS = 0;     // S_q at kTmemS + 128 q
    static constexpr int kTmemO = 256;   // O_q at kTmemO + 128 q
    static_assert(2 * kNumBars + kSchedDepth <= 2 * 64, "barrier area (barriers and the unit ring)");
};

struct WorkItem {
    SeqItem si;       // the (sequence, head) slice
    int T;            // its number of 128-row tiles
    int m;            // Q tile pair index
    int t0, t1;       // Q tile indices
    int n0, n1;       // number of KV tiles for each Q tile
};

// Work list.  Causal: units of two Q tile pairs of one head, m and M-1-m, longest first.  The
// pair m meets 2m+1 and 2m+2 key/value tiles, so every unit holds the same amount of work and
// a static round-robin of units over the persistent CTAs is balanced.  Non-causal: every item
// is equally long, so each unit is one item (a finer grain shortens the tail).  Consecutive
// units share a head, so the CTAs running at one time reuse its K / V from L2.  With packed
// sequences of different lengths the units are laid out for the longest one (M pairs per
// slice) and the items past the end of a shorter sequence are skipped.
__device__ __forceinline__ int fwd_units_per_head(int M, int causal) { return causal ? (M + 1) / 2 : M; }

template <bool kTM>
__device__ __forceinline__ bool fwd_item(int u, int s, int M, int causal, const SeqDesc& seq, WorkItem& w) {
    const int uph = fwd_units_per_head(M, causal);
    const int mp = u % uph;
    int m;
    if (causal) {
        const int ml = M - 1 - mp;
        if (s == 1 && ml == mp) return false;
        m = s ? mp : ml;
    } else {
        if (s == 1) return false;
        m = M - 1 - mp;
    }
    seq_item<kTM>(seq, u / uph, w.si);
    w.T = (w.si.len + 127) / 128;
    w.m = m;
    w.t0 = 2 * m;
    w.t1 = 2 * m + 1;
    if (w.t0 >= w.T) return false;  // past the end of this sequence
    w.n0 = causal ? min(w.t0 + 1, w.T) : w.T;
    w.n1 = causal ? min(w.t1 + 1, w.T) : w.T;
    return true;
}

// Consumer threads of the dynamic distribution: the three 128-thread warpgroups, the MMA warp
// and the two loader threads.
constexpr int kSchedConsumers = 3 * 128 + 32 + 2;

// This CTA's sequence of work items.  kDyn = false: units blockIdx.x, blockIdx.x + gridDim.x, ...
// (balanced when every unit holds the same work; the position is 2 unit + slot).  kDyn = true:
// the units the scheduler thread publishes through the ring, which lives in the barrier area:
// full[kSchedDepth] (one arrival, the scheduler thread), empty[kSchedDepth] (one arrival per
// consumer thread) and the slot words themselves.  A consumer thread holds the entry of its
// current unit until it takes the next one, so the unit index can be read again from shared
// memory and the whole position is one register: 4 (entries taken) + (next item of the unit,
// 2 = none left).  Every consumer thread releases entries itself (no warp-collective step, so a
// thread that has stopped early cannot hold up its warp).  next() is false at the end of the
// work, or when a wait gave up.
template <bool kDyn>
struct FwdIter;

template <>
struct FwdIter<false> {
    int pos = 2 * (int)blockIdx.x;
    template <bool kTM, class L>
    __device__ bool next(WorkItem& w, int M, int causal, const SeqDesc& seq, int n_units, uint64_t*,
                         const WaitGuard&, int) {
        for (;;) {
            const int u = pos >> 1, s = pos & 1;
            if (u >= n_units) return false;
            pos = s ? 2 * (u + (int)gridDim.x) : pos + 1;
            if (fwd_item<kTM>(u, s, M, causal, seq, w)) return true;
        }
    }
};

template <>
struct FwdIter<true> {
    uint32_t st = 2;
    template <bool kTM, class L>
    __device__ bool next(WorkItem& w, int M, int causal, const SeqDesc& seq, int, uint64_t* bars, const WaitGuard& g,
                         int code) {
        volatile int* ring = reinterpret_cast<volatile int*>(bars) + L::kSchedSlotWord;
        for (;;) {
            const uint32_t k = st >> 2, s = st & 3;
            if (s < 2) {
                ++st;
                if (fwd_item<kTM>(ring[(k - 1) % kSchedDepth], (int)s, M, causal, seq, w)) return true;
                continue;
            }
            if (k > 0) mbar_arrive(&bars[L::kBarSchedEmpty + (k - 1) % kSchedDepth]);
            if (!mbar_wait(&bars[L::kBarSchedFull + k % kSchedDepth], (k / kSchedDepth) & 1, g, code)) return false;
            if (ring[k % kSchedDepth] < 0) return false;
            st = 4 * (k + 1);
        }
    }
    // The item next() returned last, expanded again (lets a role keep only part of it live).
    template <bool kTM, class L>
    __device__ void current(WorkItem& w, int M, int causal, const SeqDesc& seq, uint64_t* bars) const {
        const volatile int* ring = reinterpret_cast<volatile int*>(bars) + L::kSchedSlotWord;
        fwd_item<kTM>(ring[((st >> 2) - 1) % kSchedDepth], (int)(st & 3) - 1, M, causal, seq, w);
    }
};

template <int D, bool BF16, bool kTM, bool kDyn>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o_out,
                float* __restrict__ lse_out, const SeqDesc seq, float scale, int causal,
                unsigned int* __restrict__ sched, int* error) {
    using L = FwdLayout<D>;
    // K/V ring tokens come in the order K_0, then V_j, K_{j+1} per step (V_{n-1}, K_0 of the next
    // item at an item boundary).  With the static work list the loader knows where the work ends,
    // so it signals each (V_j, following K) pair on one barrier, that of V_j's slot, and the MMA
    // warp takes one wait per step instead of two.  The pair is released the same way, with one
    // commit on V_j's empty barrier once both tiles have been read (for V_{n-1}, K_0 of the next
    // item: after that item's first S products); the loader waits on it for both slots.
    constexpr bool kPairKV = !kDyn;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Align the dynamic shared memory base to 1024 bytes (128B-swizzle atoms).
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kAux);
    float* scale_buf = reinterpret_cast<float*>(smem + L::kScaleOff);
    float* fin_l = reinterpret_cast<float*>(smem + L::kFinLOff);
    float* fin_m = reinterpret_cast<float*>(smem + L::kFinMOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = (seq.N + 127) / 128;  // tiles of the longest sequence (the last one may be ragged)
    const int M = (T + 1) / 2;
    const int n_units = seq.B * seq.H * fwd_units_per_head(M, causal);

    if (threadIdx.x == 0) {
        mbar_init(&bars[L::kBarQFull], 1);
        mbar_init(&bars[L::kBarQEmpty], 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bars[L::kBarKVFull + s], 1);
            mbar_init(&bars[L::kBarKVEmpty + s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bars[L::kBarSFull + q], 1);
            mbar_init(&bars[L::kBarPVReady + q], 256);  // 128 softmax + 128 correction threads
            mbar_init(&bars[L::kBarODone + q], 1);
            mbar_init(&bars[L::kBarStats + q], 128);
            mbar_init(&bars[L::kBarFin + 2 * q + 0], 128);
            mbar_init(&bars[L::kBarFin + 2 * q + 1], 128);
        }
        mbar_init(&bars[L::kBarTeardown], 1);
        if (kDyn) {
            for (int i = 0; i < kSchedDepth; ++i) {
                mbar_init(&bars[L::kBarSchedFull + i], 1);
                mbar_init(&bars[L::kBarSchedEmpty + i], kSchedConsumers);
            }
        }
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
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard guard{abort_flag, error, kWaitLimitNs};
    const float scale_log2 = scale * kLog2e;
    const int wg = warp >> 2;

    if (wg == 0 || wg == 1) {
        // ------------------------------------------------------------ softmax
        regs_inc<176>();
        const int q = wg;
        const int row = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + L::kTmemS + 128 * q;
        uint32_t s_phase = 0;
        int k = 0;
        bool ok = true;
        WorkItem w;
        for (FwdIter<kDyn> itr; ok && itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutSoftmax); ++k) {
            const int t = q ? w.t1 : w.t0;
            const int n = q ? w.n1 : w.n0;
            const int diag = (causal && t < w.T) ? t : -1;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < n; ++j) {
                if (!mbar_wait(&bars[L::kBarSFull + q], s_phase, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                s_phase ^= 1;
                tc_fence_after();
                uint32_t s[128];
                tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                tmem_wait_ld();
                // Masked columns c > lim: on the diagonal tile a key index above the query index
                // (aligned top-left causal mask); in a ragged last tile the keys past the end of the
                // sequence (zeros, or rows of the next sequence).
                int lim = 127;
                if (j == diag) lim = row;
                if (j == w.T - 1) lim = min(lim, w.si.len - 1 - j * 128);
                if (lim < 127) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > lim) s[c] = __float_as_uint(-INFINITY);
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    mx0 = fmax3(mx0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
                    mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
                    mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
                }
                const float tile_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
                float alpha = 1.f;
                if (j == 0) {
                    m_run = tile_max;
                } else if (tile_max - m_run > kRescaleThreshold) {
                    alpha = ex2_ftz(m_run - tile_max);
                    l_run *= alpha;
                    m_run = tile_max;
                }
                scale_buf[q * 128 + row] = alpha;
                mbar_arrive(&bars[L::kBarStats + q]);

                // p = 2^(s * scale * log2(e) - m), rounded to 16 bits for the PV MMA; the row sum
                // l adds the FP32 values (it gives L and normalises O).
                const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
                const uint64_t nm2 = f2_pack(-m_run, -m_run);
                uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[32 * h + 2 * c]),
                                                          __uint_as_float(s[32 * h + 2 * c + 1])), sl2, nm2);
                        float x0, x1;
                        f2_unpack(x, x0, x1);
                        const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
                        pk[c] = pack2<BF16>(p0, p1);
                        if (c & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
                        else acc0 = f2_add(acc0, f2_pack(p0, p1));
                    }
                    tmem_st16(s_addr + 16 * h, pk);
                }
                float sa, sb, sc, sd;
                f2_unpack(acc0, sa, sb);
                f2_unpack(acc1, sc, sd);
                l_run += (sa + sb) + (sc + sd);
                if (j == n - 1) {
                    const int b = k & 1;
                    fin_l[(b * 2 + q) * 128 + row] = l_run;
                    fin_m[(b * 2 + q) * 128 + row] = m_run;
                    mbar_arrive(&bars[L::kBarFin + 2 * q + b]);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[L::kBarPVReady + q]);
            }
        }
    } else if (wg == 2) {
        // ------------------------------------------------ correction + epilogue
        regs_dec<72>();
        const int row = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        // Wait parities (bit q for Stats[q], bit 2 + q for ODone[q]) and, from bit 4 up, the
        // number of items done: one register.
        uint32_t ph = 0;
        bool ok = true;
        // O rows start at multiples of 128 bytes, so 32-byte stores need only a 32-byte aligned base
        // (the interface guarantees 16).  The dynamically scheduled (packed) instance keeps 16-byte
        // stores: with the wider ones it measured 1091 against 1134 TFLOPS, as its code placement
        // moved.
        const bool o_al32 = !kDyn && (reinterpret_cast<uintptr_t>(o_out) & 31u) == 0;
        FwdIter<kDyn> itr;
        for (WorkItem w0; ok && itr.template next<kTM, L>(w0, M, causal, seq, n_units, bars, guard, kDevTimeoutCorr);
             ph += 16) {
            // With the dynamic distribution only the tile counts stay live through the loop and the
            // epilogue expands the item again (the warpgroup has 72 registers).
            const int n0 = w0.n0, n1 = w0.n1;
            for (int j = 0; j < n1 && ok; ++j) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = q ? n1 : n0;
                    if (j >= n) continue;
                    if (!mbar_wait(&bars[L::kBarStats + q], (ph >> q) & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                    ph ^= 1u << q;
                    const float alpha = scale_buf[q * 128 + row];
                    if (j > 0) {
                        if (!mbar_wait(&bars[L::kBarODone + q], (ph >> (2 + q)) & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                        ph ^= 4u << q;
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
                            const uint32_t o_addr = tmem + lane_base + L::kTmemO + 128 * q;
#pragma unroll 1
                            for (int c = 0; c < D; c += 32) {
                                uint32_t r[32];
                                tmem_ld32(o_addr + c, r);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                                tmem_st32(o_addr + c, r);
                            }
                            tmem_wait_st();
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&bars[L::kBarPVReady + q]);
                }
            }
            if (!ok) break;
            // epilogue: O = O / l -> 16-bit, L = (m + log2 l) ln 2
            WorkItem w;
            if constexpr (kDyn) itr.template current<kTM, L>(w, M, causal, seq, bars);
            else w = w0;
            for (int q = 0; q < 2 && ok; ++q) {
                const uint32_t b = (ph >> 4) & 1;
                if (!mbar_wait(&bars[L::kBarODone + q], (ph >> (2 + q)) & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                ph ^= 4u << q;
                if (!mbar_wait(&bars[L::kBarFin + 2 * q + b], (ph >> 5) & 1, guard, kDevTimeoutCorr)) { ok = false; break; }
                tc_fence_after();
                const float l = fin_l[(b * 2 + q) * 128 + row];
                const float mrow = fin_m[(b * 2 + q) * 128 + row];
                const int t = q ? w.t1 : w.t0;
                const int grow = t * 128 + row;
                const float inv_l = 1.f / l;
                const uint32_t o_addr = tmem + lane_base + L::kTmemO + 128 * q;
                uint8_t* dst = reinterpret_cast<uint8_t*>(o_out) + seq_row_offset<kTM>(seq, w.si, grow, D) * 2;
                // d = 128, [B, H, N, d]: 16 columns per TMEM load, two loads in flight: the next
                // chunk is loaded while this one is scaled, rounded and stored, so the load latency
                // is paid once per tile rather than once per chunk (the next item's first PV_q
                // waits for this epilogue to have read O_q; +1.1 to +1.5 % on the forward).
                auto store16 = [&](const uint32_t (&r)[16], int c) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pk[e] = pack2<BF16>(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
                    if (grow < w.si.len) {
                        // A thread writes its own row, so a warp store touches 32 rows; 32-byte
                        // stores fill whole sectors and halve the store instructions (measured:
                        // forward 1326 -> 1361 TFLOPS at causal B=8 H=16 N=4096 d=128).
                        if (o_al32) {
                            st_global_v8(dst + c * 2, pk);
                        } else {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 2);
                            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                };
                if constexpr (!kTM && D == 64) {
                    // two 32-column chunks, one load in flight (measured faster at d = 64 than the
                    // double-buffered 16-column loads: 0.191 against 0.194 ms, causal B=4 H=16 N=4096)
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + c, r);
                        tmem_wait_ld();
                        store16(*reinterpret_cast<const uint32_t(*)[16]>(&r[0]), c);
                        store16(*reinterpret_cast<const uint32_t(*)[16]>(&r[16]), c + 16);
                    }
                } else if constexpr (!kTM) {
                    uint32_t ra[16], rb[16];
                    tmem_ld16(o_addr, ra);
                    tmem_wait_ld();
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        tmem_ld16(o_addr + c + 16, rb);
                        store16(ra, c);
                        tmem_wait_ld();
                        if (c + 32 < D) tmem_ld16(o_addr + c + 32, ra);
                        store16(rb, c + 16);
                        tmem_wait_ld();
                    }
                } else {
                    // token-major rows need more address registers: one load in flight keeps the
                    // warpgroup inside its 72 registers
#pragma unroll 1
                    for (int c = 0; c < D; c += 16) {
                        uint32_t r[16];
                        tmem_ld16(o_addr + c, r);
                        tmem_wait_ld();
                        store16(r, c);
                    }
                }
                if (grow < w.si.len) lse_out[seq_lse_index<kTM>(seq, w.si, grow)] = (mrow + log2f(l)) * kLn2;
                tc_fence_before();
            }
        }
    } else {
        regs_dec<88>();  // warps 12-15; the split 2x176 + 72 + 88 warpgroups uses 65536 registers
        if (warp == 12) {
            // ------------------------------------------------------------ MMA issuer (the whole warp; lane 0 issues)
            constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16, false, false);
            constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16, false, true);
            const uint32_t q_base[2] = {smem_u32(smem + L::kQ0), smem_u32(smem + L::kQ1)};
            const uint32_t kv_base = smem_u32(smem + L::kKV);
            uint32_t tok = 0, q_phase = 0, pv_phase[2] = {0, 0};
            bool ok = true;
            // S_q = Q_q K^T (K-major operands, D / 16 steps) and O_q += P_q V (P packed in S_q's
            // first 64 columns, 8 columns per step; V read MN-major), each one chain of MMAs.
            auto issue_qk = [&](int q, uint32_t slot) {
                const uint32_t d_tmem = tmem + L::kTmemS + 128 * q;
                const uint64_t a = sdesc_sw128(q_base[q], 16, 1024);
                const uint64_t b = sdesc_sw128(kv_base + slot * L::kTile, 16, 1024);
                if constexpr (D == 128)
                    warp_mma_ss8<GB300_KMAJ_OFFS(kPanelBytes), GB300_KMAJ_OFFS(kPanelBytes)>(d_tmem, a, b, kIdescQK, 0);
                else
                    warp_mma_ss4<2, 4, 6, 2, 4, 6>(d_tmem, a, b, kIdescQK, 0);
            };
            auto issue_pv = [&](int q, uint32_t slot, bool acc) {
                const uint32_t d_tmem = tmem + L::kTmemO + 128 * q;
                const uint32_t p_tmem = tmem + L::kTmemS + 128 * q;
                const uint64_t b = sdesc_sw128(kv_base + slot * L::kTile, kPanelBytes, 1024);
                warp_mma_ts8<8, 16, 24, 32, 40, 48, 56, GB300_MNMAJ_OFFS>(d_tmem, p_tmem, b, kIdescPV, acc ? 1u : 0u);
            };
            auto wait_kv = [&](uint32_t& slot) -> bool {
                slot = tok % L::kStages;
                const bool r = warp_mbar_wait(&bars[L::kBarKVFull + slot], (tok / L::kStages) & 1, guard, kDevTimeoutMma);
                ++tok;
                tc_fence_after();
                return r;
            };
            int pending = -1;  // kPairKV: slot of a V whose pair ends with the next item's K_0
            WorkItem w;
            for (FwdIter<kDyn> itr; ok && itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutMma);) {
                if (!warp_mbar_wait(&bars[L::kBarQFull], q_phase, guard, kDevTimeoutMma)) { ok = false; break; }
                q_phase ^= 1;
                tc_fence_after();
                uint32_t kslot;
                if (kPairKV && tok > 0) {
                    kslot = tok++ % L::kStages;  // landed with the previous item's last V
                } else if (!wait_kv(kslot)) {
                    ok = false;
                    break;
                }
                issue_qk(0, kslot);
                warp_mma_commit(&bars[L::kBarSFull + 0]);
                issue_qk(1, kslot);
                warp_mma_commit(&bars[L::kBarSFull + 1]);
                warp_mma_commit(&bars[L::kBarKVEmpty + (kPairKV && pending >= 0 ? (uint32_t)pending : kslot)]);
                pending = -1;
                // Q is read by the S MMAs only: the Q buffers are released after the item's last
                // S (S_1(n1 - 1); S_0's last comes no later), so that the next item's Q loads
                // while this item's last PVs and epilogue run.
                if (w.n1 == 1) warp_mma_commit(&bars[L::kBarQEmpty]);
                for (int j = 0; j < w.n1 && ok; ++j) {
                    uint32_t vslot;
                    if (!wait_kv(vslot)) { ok = false; break; }  // kPairKV: V_j and the K after it
                    bool have_k = false;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int n = q ? w.n1 : w.n0;
                        if (j >= n) continue;
                        if (!warp_mbar_wait(&bars[L::kBarPVReady + q], pv_phase[q], guard, kDevTimeoutMma)) { ok = false; break; }
                        pv_phase[q] ^= 1;
                        tc_fence_after();
                        issue_pv(q, vslot, j > 0);
                        warp_mma_commit(&bars[L::kBarODone + q]);
                        if (j + 1 < n) {
                            if (!have_k) {
                                if (kPairKV) kslot = tok++ % L::kStages;
                                else if (!wait_kv(kslot)) { ok = false; break; }
                                have_k = true;
                            }
                            issue_qk(q, kslot);
                            warp_mma_commit(&bars[L::kBarSFull + q]);
                            if (q == 1 && j + 2 == w.n1) warp_mma_commit(&bars[L::kBarQEmpty]);
                        }
                    }
                    if (!ok) break;
                    if constexpr (kPairKV) {
                        if (have_k) warp_mma_commit(&bars[L::kBarKVEmpty + vslot]);
                        else pending = (int)vslot;  // released after the next item's K_0 is read
                    } else {
                        warp_mma_commit(&bars[L::kBarKVEmpty + vslot]);
                        if (have_k) warp_mma_commit(&bars[L::kBarKVEmpty + kslot]);
                    }
                }
            }
            if (kPairKV && pending >= 0) warp_mma_commit(&bars[L::kBarKVEmpty + pending]);
            // Every MMA issued above completes before TMEM is released.
            warp_mma_commit(&bars[L::kBarTeardown]);
            mbar_wait_drain(&bars[L::kBarTeardown], 0, kWaitLimitNs);
        } else if (warp == 14 && lane == 0) {
            // ------------------------------------------------------------ TMA producer: Q tiles
            // (its own warp, so that the K/V stream below never waits for a Q buffer to free up)
            int k = 0;
            bool ok = true;
            int last_q_item = -1;
            WorkItem w;
            for (FwdIter<kDyn> itr; ok && itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutLoad); ++k) {
                if (k > 0 && !mbar_wait(&bars[L::kBarQEmpty], (k - 1) & 1, guard, kDevTimeoutLoad)) { ok = false; break; }
                mbar_arrive_expect_tx(&bars[L::kBarQFull], 2 * L::kTile);
                last_q_item = k;
#pragma unroll
                for (int p = 0; p < L::kPanels; ++p) {
                    seq_tma_load<kTM>(smem + L::kQ0 + p * kPanelBytes, &tm_q, &bars[L::kBarQFull], w.si, 64 * p, w.t0 * 128);
                    seq_tma_load<kTM>(smem + L::kQ1 + p * kPanelBytes, &tm_q, &bars[L::kBarQFull], w.si, 64 * p, w.t1 * 128);
                }
            }
            // Let every copy issued above land before shared memory is released.
            if (last_q_item >= 0) mbar_wait_drain(&bars[L::kBarQFull], last_q_item & 1, kWaitLimitNs);
        } else if (warp == 13 && lane == 0) {
            // ------------------------------------------------------------ TMA producer: K/V ring
            uint32_t tok = 0;
            bool ok = true;
            WorkItem w;
            FwdIter<kDyn> itr;
            bool more = itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutLoad);
            while (ok && more) {
                const WorkItem cur = w;
                // kPairKV: whether a K follows this item's last V (the static list is read one item
                // ahead; the dynamic one is not, its next unit is taken only when needed)
                if constexpr (kPairKV) more = itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutLoad);
                for (int j = 0; j < cur.n1 && ok; ++j) {
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        const uint32_t slot = tok % L::kStages;
                        // the previous tile in this slot must have been read.  kPairKV: a pair's
                        // first slot waits for the release of the pair there before (both slots),
                        // a second slot only where it last held the lone first K (token 0).
                        const bool wait_empty = tok >= (uint32_t)L::kStages &&
                                                (!kPairKV || (tok & 1) || tok == (uint32_t)L::kStages);
                        if (wait_empty &&
                            !mbar_wait(&bars[L::kBarKVEmpty + slot], ((tok / L::kStages) - 1) & 1, guard, kDevTimeoutLoad)) {
                            ok = false;
                            break;
                        }
                        // the barrier this tile lands on: its own, or (kPairKV, a K after the first
                        // token) that of the V before it, which expects both tiles
                        uint32_t fslot = slot;
                        if (!kPairKV || tok == 0) {
                            mbar_arrive_expect_tx(&bars[L::kBarKVFull + slot], L::kTile);
                        } else if (tok & 1) {
                            const bool pair = more || j + 1 < cur.n1;
                            mbar_arrive_expect_tx(&bars[L::kBarKVFull + slot], pair ? 2 * L::kTile : L::kTile);
                        } else {
                            fslot = (tok - 1) % L::kStages;
                        }
                        const CUtensorMap* map = which ? &tm_v : &tm_k;
#pragma unroll
                        for (int p = 0; p < L::kPanels; ++p)
                            seq_tma_load<kTM>(smem + L::kKV + slot * L::kTile + p * kPanelBytes, map,
                                         &bars[L::kBarKVFull + fslot], cur.si, 64 * p, j * 128);
                        ++tok;
                    }
                }
                if (!ok) break;
                if constexpr (!kPairKV) more = itr.template next<kTM, L>(w, M, causal, seq, n_units, bars, guard, kDevTimeoutLoad);
            }
            // Let every copy issued above land before shared memory is released (kPairKV: the
            // second tile of a pair lands on the first one's barrier).
            for (uint32_t t = (tok > (uint32_t)L::kStages ? tok - L::kStages : 0); t < tok; ++t)
                if (!kPairKV || t == 0 || (t & 1))
                    mbar_wait_drain(&bars[L::kBarKVFull + t % L::kStages], (t / L::kStages) & 1, kWaitLimitNs);
        } else if (kDyn && warp == 15 && lane == 0) {
            // ------------------------------------------------------------ scheduler
            // It waits with a sleep between polls: its warp shares a scheduler with softmax warps.
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
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool BF16, bool kTM, bool kDyn>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
    using L = FwdLayout<D>;
    const int smem_bytes = L::kBytes + 1024;  // + alignment slack
    auto kern = attn_fwd_kernel<D, BF16, kTM, kDyn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    const int T = (a.N + 127) / 128;
    const int M = (T + 1) / 2;
    const long n_units = (long)a.BH * (a.causal ? (M + 1) / 2 : M);
    const int grid = (int)(n_units < a.num_sms ? n_units : a.num_sms);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, kThreads, smem_bytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.seq, a.scale, a.causal,
                                                  a.sched, a.error);
    return cudaGetLastError();
}

template <bool kTM, bool kDyn>
cudaError_t launch_fwd_l(const FwdArgs& a, cudaStream_t stream) {
    if (a.d == 128)
        return a.fp16 ? launch_fwd_t<128, false, kTM, kDyn>(a, stream) : launch_fwd_t<128, true, kTM, kDyn>(a, stream);
    if (a.d == 64)
        return a.fp16 ? launch_fwd_t<64, false, kTM, kDyn>(a, stream) : launch_fwd_t<64, true, kTM, kDyn>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

// Row layout and work distribution: [B, H, N, d] and BSHD hold sequences of one length, whose
// units all carry the same work, so the static distribution is balanced and costs nothing;
// packed sequences of different lengths take units from the launch's work counter.
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
    if (!a.seq.token_major) return launch_fwd_l<false, false>(a, stream);
    return a.seq.cu ? launch_fwd_l<true, true>(a, stream) : launch_fwd_l<true, false>(a, stream);
}

}  // namespace gb300
