// Single-query (decode) attention against a key/value cache, for sm_103a.
//
// Per (batch b, query head h): o = softmax(scale q K^T) V over the cached keys
// 0 .. len_b - 1 and L = log sum exp(scale q K^T) -- the forward equations of
// "Writing Speed-of-Light Attention Backward Kernel for 5090 in CUDA" (section
// "Mathematical Formulation") with one query row and no mask.  The
// flash_attention_cuda README lists a KV-cache decode kernel as the missing
// piece for generation ("a different, memory-bound problem").
//
// The work is HBM-bound (every cached key and value is read once, a few FLOPs
// per byte), so the design streams K and V at full bandwidth and spends tensor
// cores freely:
//  * grouped queries: the G = Hq / Hkv query heads that share KV head
//    (b, hkv) are the rows of one zero-padded 128-row Q tile, so one
//    S = Q K^T MMA (tcgen05, M = 128) serves all of them and K / V are read
//    once per group;
//  * split KV: the keys of a group are cut into chunks of whole 128-key tiles,
//    at least 512 KB of K / V (1024 keys at d = 128, 2048 at d = 64), their
//    length chosen per launch so that the (group, chunk) items fill the
//    persistent grid (one CTA per SM) in whole waves, so that even a small
//    batch covers every SM with little tail; each item writes its
//    chunk's O (normalised) and L, and a second kernel combines the chunks:
//    L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s;
//  * per chunk the pipeline of the forward kernel, reduced to one Q tile: a
//    TMA producer streams 128-key K and V tiles through a ring (4 slots at
//    d = 128, 8 at d = 64: 128 KB in flight per SM either way), the MMA
//    warp computes S into one of two TMEM buffers while the softmax warps turn
//    the other into P (16-bit, in TMEM over S), then O += P V (TS-MMA).  The
//    running max uses the lazy rescale of the forward (threshold 8, base 2).
//
// CTA layout (192 threads): warps 0-3 softmax and epilogue (thread = Q row =
// query head of the group; warps whose rows are all >= G idle), warp 4 MMA
// issuer (whole warp, lane 0 issues; owns TMEM), warp 5 TMA producer.
// TMEM: S0 [0,128), S1 [128,256), O [256, 256 + d).
#include "attn_internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kDecThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kPanelBytes = 128 * 128;

template <int D>
struct DecLayout {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kStages = D == 128 ? 4 : 8;  // 128 KB of K/V tiles in flight either way
    static constexpr int kQ = 0;          // [2]: non-empty item i uses slot i % 2, so the next
    static constexpr int kKV = 2 * kTile;  // item's Q loads while this one runs
    static constexpr int kAux = kKV + kStages * kTile;
    static constexpr int kBarQFull = 0, kBarQEmpty = 2;  // [2] each
    static constexpr int kBarKVFull = 4;
    static constexpr int kBarKVEmpty = kBarKVFull + kStages;
    static constexpr int kBarSFull = kBarKVEmpty + kStages;  // [2]: tile g uses buffer g % 2
    static constexpr int kBarPReady = kBarSFull + 2;         // [2]
    static constexpr int kBarODone = kBarPReady + 2;         // [2]: PV(g) commits to ODone[g % 2]
    static constexpr int kBarOFree = kBarODone + 2;          // O read out by the epilogue
    static constexpr int kBarTeardown = kBarOFree + 1;
    static constexpr int kNumBars = kBarTeardown + 1;
    static constexpr int kMiscOff = kAux + kNumBars * 8;
    static constexpr int kBytes = kMiscOff + 16;
    static constexpr int kTmemS = 0, kTmemO = 256;
};

// Work item u = (group bh, chunk s): keys [k0, k1) of the group's cache, n_tiles 128-key tiles.
struct DecItem {
    int bh, s, k0, k1, n_tiles;
};

__device__ __forceinline__ void dec_item(int u, int splits, int chunk, int Hkv, int Nmax, const int* seqlens,
                                         int* error, bool report, DecItem& w) {
    w.bh = u / splits;
    w.s = u - w.bh * splits;
    int len = Nmax;
    if (seqlens != nullptr) {
        len = __ldg(seqlens + w.bh / Hkv);
        if (len < 0 || len > Nmax) {  // not a valid cache length: nothing of this batch is read
            if (report) atomicCAS(error, 0, kDevBadSeqLen);
            len = 0;
        }
    }
    w.k0 = w.s * chunk;
    w.k1 = min(w.k0 + chunk, len);
    w.n_tiles = w.k1 > w.k0 ? (w.k1 - w.k0 + 127) / 128 : 0;
}

// Persistent: CTA c takes items c, c + gridDim.x, ...  Tile and ring counters run on across
// items, so every barrier phase below is a function of a global tile (g) or item count.
template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads, 1)
attn_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const int* __restrict__ seqlens,
                   float* __restrict__ part_o, float* __restrict__ part_l, void* __restrict__ o_out,
                   float* __restrict__ lse_out, int Hkv, int G, int Nmax, int splits, int chunk, int n_items,
                   float scale, int* error) {
    using L = DecLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kAux);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int active_warps = min(4, (G + 31) / 32);  // softmax warps holding at least one real row

    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bars[L::kBarQFull + q], 1);
            mbar_init(&bars[L::kBarQEmpty + q], 1);
        }
        for (int st = 0; st < L::kStages; ++st) {
            mbar_init(&bars[L::kBarKVFull + st], 1);
            mbar_init(&bars[L::kBarKVEmpty + st], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bars[L::kBarSFull + q], 1);
            mbar_init(&bars[L::kBarPReady + q], 32 * active_warps);  // every thread of the active warps
            mbar_init(&bars[L::kBarODone + q], 1);
        }
        mbar_init(&bars[L::kBarOFree], 32 * active_warps);
        mbar_init(&bars[L::kBarTeardown], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 4) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard guard{abort_flag, error, kWaitLimitNs};

    if (warp < 4) {
        // ------------------------------------------------------------ softmax + epilogue
        if (warp < active_warps) {
            const int row = threadIdx.x;  // query head (row) of the group
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
            const float scale_log2 = scale * kLog2e;
            uint32_t gt = 0;  // global index of the item's first tile
            bool ok = true;
            for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x) {
                DecItem w;
                dec_item(u, splits, chunk, Hkv, Nmax, seqlens, error, threadIdx.x == 0, w);
                float* po = part_o + (size_t)u * G * D;
                float* pl = part_l + (size_t)u * G;
                // one chunk per group: this item's result is the final one (query head u G + row),
                // written here in 16 bits, and no combination kernel runs
                uint8_t* od = static_cast<uint8_t*>(o_out) + ((size_t)u * G + row) * D * 2;
                if (w.n_tiles == 0) {
                    // empty chunk: weight exp(-inf) = 0 in the combination (an empty cache: O = 0, L = -inf)
                    if (row < G) {
                        if (splits == 1) {
                            for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(od + c * 2) = make_uint4(0, 0, 0, 0);
                            lse_out[(size_t)u * G + row] = -INFINITY;
                        } else {
                            pl[row] = -INFINITY;
                            for (int c = 0; c < D; c += 4)
                                *reinterpret_cast<float4*>(po + (size_t)row * D + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    continue;
                }
                float m_run = -INFINITY, l_run = 0.f;
                for (int j = 0; j < w.n_tiles; ++j) {
                    const uint32_t g = gt + j;
                    const int buf = g & 1;
                    if (!warp_mbar_wait(&bars[L::kBarSFull + buf], (g >> 1) & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t s_addr = tmem + lane_base + L::kTmemS + 128 * buf;
                    uint32_t sv[128];
                    tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[64]));
                    tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[96]));
                    tmem_wait_ld();
                    // keys past the chunk (the next chunk's, past the cache length, or the zero fill)
                    const int lim = min(127, w.k1 - 1 - (w.k0 + 128 * j));
                    if (lim < 127) {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (c > lim) sv[c] = __float_as_uint(-INFINITY);
                    }
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 128; c += 4) {
                        mx0 = fmax3(mx0, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
                        mx1 = fmax3(mx1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
                    }
                    const float tile_max = fmaxf(mx0, mx1) * scale_log2;
                    float alpha = 1.f;
                    if (j == 0) {
                        m_run = tile_max;
                    } else if (tile_max - m_run > kRescaleThreshold) {
                        alpha = ex2_ftz(m_run - tile_max);
                        l_run *= alpha;
                        m_run = tile_max;
                    }
                    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        // O holds tiles < g; PV(g-1) is the newest that can still be running (the
                        // S(g) waited for above was committed after PV(g-2)), and the previous phase
                        // of its barrier (PV(g-3)) is complete.
                        const uint32_t p = g - 1;
                        if (!warp_mbar_wait(&bars[L::kBarODone + (p & 1)], (p >> 1) & 1, guard, kDevTimeoutSoftmax)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t o_addr = tmem + lane_base + L::kTmemO;
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
                    const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
                    const uint64_t nm2 = f2_pack(-m_run, -m_run);
                    uint64_t acc = 0;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[32 * h + 2 * c]),
                                                              __uint_as_float(sv[32 * h + 2 * c + 1])), sl2, nm2);
                            float x0, x1;
                            f2_unpack(x, x0, x1);
                            const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
                            pk[c] = pack2<BF16>(p0, p1);
                            acc = f2_add(acc, f2_pack(p0, p1));
                        }
                        tmem_st16(s_addr + 16 * h, pk);
                    }
                    float sa, sb;
                    f2_unpack(acc, sa, sb);
                    l_run += sa + sb;
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars[L::kBarPReady + buf]);
                }
                if (!ok) break;
                // epilogue: the item's last PV is done once its barrier phase completes (the one
                // before it, two tiles back, is complete since the last S(g) was waited for)
                const uint32_t p = gt + w.n_tiles - 1;
                if (!warp_mbar_wait(&bars[L::kBarODone + (p & 1)], (p >> 1) & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                tc_fence_after();
                const float inv_l = 1.f / l_run;
                const uint32_t o_addr = tmem + lane_base + L::kTmemO;
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + c, r);
                    tmem_wait_ld();
                    if (row < G && splits == 1) {
                        uint4* dst = reinterpret_cast<uint4*>(od + c * 2);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pack2<BF16>(__uint_as_float(r[8 * e]) * inv_l, __uint_as_float(r[8 * e + 1]) * inv_l),
                                                pack2<BF16>(__uint_as_float(r[8 * e + 2]) * inv_l, __uint_as_float(r[8 * e + 3]) * inv_l),
                                                pack2<BF16>(__uint_as_float(r[8 * e + 4]) * inv_l, __uint_as_float(r[8 * e + 5]) * inv_l),
                                                pack2<BF16>(__uint_as_float(r[8 * e + 6]) * inv_l, __uint_as_float(r[8 * e + 7]) * inv_l));
                    } else if (row < G) {
                        float4* dst = reinterpret_cast<float4*>(po + (size_t)row * D + c);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv_l, __uint_as_float(r[4 * e + 1]) * inv_l,
                                                 __uint_as_float(r[4 * e + 2]) * inv_l,
                                                 __uint_as_float(r[4 * e + 3]) * inv_l);
                    }
                }
                if (row < G) {
                    const float lrow = (m_run + log2f(l_run)) * kLn2;
                    if (splits == 1) lse_out[(size_t)u * G + row] = lrow;
                    else pl[row] = lrow;
                }
                tc_fence_before();
                mbar_arrive(&bars[L::kBarOFree]);  // O may now be overwritten by the next item
                gt += w.n_tiles;
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer (whole warp)
        constexpr uint32_t kIdescQK = idesc_f16(128, 128, BF16, false, false);
        constexpr uint32_t kIdescPV = idesc_f16(128, D, BF16, false, true);
        const uint32_t q_base0 = smem_u32(smem + L::kQ);
        uint32_t q_base = q_base0;
        const uint32_t kv_base = smem_u32(smem + L::kKV);
        bool ok = true;
        // The ring's tokens are K(0) V(0) K(1) V(1) ... over the global tile index g: K(g) is token
        // 2g, V(g) token 2g + 1.
        auto wait_tok = [&](uint32_t t) -> bool {
            const bool r = warp_mbar_wait(&bars[L::kBarKVFull + t % L::kStages], (t / L::kStages) & 1, guard,
                                          kDevTimeoutMma);
            tc_fence_after();
            return r;
        };
        auto issue_s = [&](int buf, uint32_t slot) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
                warp_mma_ss(tmem + L::kTmemS + 128 * buf, sdesc_sw128(q_base + off, 16, 1024),
                            sdesc_sw128(kv_base + slot * L::kTile + off, 16, 1024), kIdescQK, kk > 0);
            }
        };
        auto issue_pv = [&](int buf, uint32_t slot, bool acc) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bd = sdesc_sw128(kv_base + slot * L::kTile + kk * 2048, kPanelBytes, 1024);
                warp_mma_ts(tmem + L::kTmemO, tmem + L::kTmemS + 128 * buf + kk * 8, bd, kIdescPV,
                            (acc || kk > 0) ? 1u : 0u);
            }
        };
        uint32_t gt = 0, qi = 0;  // global tile index of the item's first tile; non-empty items so far
        for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x) {
            DecItem w;
            dec_item(u, splits, chunk, Hkv, Nmax, seqlens, error, false, w);
            if (w.n_tiles == 0) continue;
            if (!warp_mbar_wait(&bars[L::kBarQFull + (qi & 1)], (qi >> 1) & 1, guard, kDevTimeoutMma)) { ok = false; break; }
            tc_fence_after();
            q_base = q_base0 + (qi & 1) * L::kTile;
            for (int j = 0; j <= w.n_tiles && ok; ++j) {
                // S(g) into buffer g % 2 as soon as K(g) is in (the buffer's previous contents,
                // P(g-2), were read by PV(g-2), issued earlier), then PV(g-1) once P(g-1) and
                // V(g-1) are ready.
                if (j < w.n_tiles) {
                    const uint32_t g = gt + j, t = 2u * g;
                    if (!wait_tok(t)) { ok = false; break; }
                    issue_s(g & 1, t % L::kStages);
                    warp_mma_commit(&bars[L::kBarSFull + (g & 1)]);
                    warp_mma_commit(&bars[L::kBarKVEmpty + t % L::kStages]);
                }
                if (j > 0) {
                    const uint32_t p = gt + j - 1, t = 2u * p + 1;
                    if (!warp_mbar_wait(&bars[L::kBarPReady + (p & 1)], (p >> 1) & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                    // the first PV of an item overwrites O: the previous item's epilogue must have
                    // read it out (its OFree phase is qi - 1)
                    if (j == 1 && qi > 0 &&
                        !warp_mbar_wait(&bars[L::kBarOFree], (qi - 1) & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                    if (!wait_tok(t)) { ok = false; break; }
                    issue_pv(p & 1, t % L::kStages, j > 1);
                    warp_mma_commit(&bars[L::kBarODone + (p & 1)]);
                    warp_mma_commit(&bars[L::kBarKVEmpty + t % L::kStages]);
                }
            }
            if (!ok) break;
            warp_mma_commit(&bars[L::kBarQEmpty + (qi & 1)]);  // every MMA that reads this Q slot is issued
            gt += w.n_tiles;
            ++qi;
        }
        warp_mma_commit(&bars[L::kBarTeardown]);
        mbar_wait_drain(&bars[L::kBarTeardown], 0, kWaitLimitNs);
    } else if (lane == 0) {
        // ------------------------------------------------------------ TMA producer (warp 5)
        uint32_t tok = 0, qi = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x) {
            DecItem w;
            dec_item(u, splits, chunk, Hkv, Nmax, seqlens, error, false, w);
            if (w.n_tiles == 0) continue;
            const uint32_t qs = qi & 1;
            if (qi >= 2 && !mbar_wait(&bars[L::kBarQEmpty + qs], ((qi >> 1) - 1) & 1, guard, kDevTimeoutLoad)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&bars[L::kBarQFull + qs], L::kTile);
#pragma unroll
            for (int p = 0; p < L::kPanels; ++p)
                tma_load_3d(smem + L::kQ + qs * L::kTile + p * kPanelBytes, &tm_q, &bars[L::kBarQFull + qs], 64 * p, 0,
                            w.bh);
            ++qi;
            for (int j = 0; j < w.n_tiles && ok; ++j) {
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint32_t slot = tok % L::kStages;
                    if (tok >= (uint32_t)L::kStages &&
                        !mbar_wait(&bars[L::kBarKVEmpty + slot], ((tok / L::kStages) - 1) & 1, guard, kDevTimeoutLoad)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[L::kBarKVFull + slot], L::kTile);
                    const CUtensorMap* map = which ? &tm_v : &tm_k;
#pragma unroll
                    for (int p = 0; p < L::kPanels; ++p)
                        tma_load_3d(smem + L::kKV + slot * L::kTile + p * kPanelBytes, map, &bars[L::kBarKVFull + slot],
                                    64 * p, w.k0 + 128 * j, w.bh);
                    ++tok;
                }
            }
        }
        // Let every copy issued above land before shared memory is released.
        for (uint32_t i = (qi > 2 ? qi - 2 : 0); i < qi; ++i)
            mbar_wait_drain(&bars[L::kBarQFull + (i & 1)], (i >> 1) & 1, kWaitLimitNs);
        for (uint32_t t = (tok > (uint32_t)L::kStages ? tok - L::kStages : 0); t < tok; ++t)
            mbar_wait_drain(&bars[L::kBarKVFull + t % L::kStages], (t / L::kStages) & 1, kWaitLimitNs);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// o[b, hkv G + r, :] and L from the chunks' partial results: one CTA of 512 threads per query
// head.  All threads first reduce the chunks' L to their maximum and the weight sum; then thread
// t adds column t % d of the chunks s = t / d, t / d + 512 / d, ... (coalesced rows of the
// partial O, several loads in flight per thread), and the 512 / d partial sums are added in
// shared memory.  Chunk counts reach the hundreds for long caches, so the chunks are spread
// over threads rather than walked by one warp.
constexpr int kCombThreads = 512;

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombThreads) attn_decode_combine_kernel(const float* __restrict__ part_o,
                                                                           const float* __restrict__ part_l,
                                                                           void* __restrict__ o, float* __restrict__ lse,
                                                                           int G, int splits) {
    constexpr int kGroups = kCombThreads / D;
    __shared__ float red[kCombThreads / 32];
    __shared__ float part[kGroups][D];
    const int row = blockIdx.x;  // query head b Hq + hkv G + r
    const int bh = row / G, r = row - bh * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* pl = part_l + (size_t)bh * splits * G + r;  // chunk s at pl[s * G]

    float m = -INFINITY;
    for (int s = tid; s < splits; s += kCombThreads) m = fmaxf(m, pl[(size_t)s * G]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float lmax = red[0];
#pragma unroll
    for (int w = 1; w < kCombThreads / 32; ++w) lmax = fmaxf(lmax, red[w]);
    __syncthreads();

    float ws = 0.f;
    if (lmax != -INFINITY)
        for (int s = tid; s < splits; s += kCombThreads) ws += __expf(pl[(size_t)s * G] - lmax);  // 0 when empty
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
    if (lane == 0) red[warp] = ws;
    __syncthreads();
    float wsum = 0.f;
#pragma unroll
    for (int w = 0; w < kCombThreads / 32; ++w) wsum += red[w];

    const int e = tid % D, grp = tid / D;
    float acc = 0.f;
    if (lmax != -INFINITY) {
        const float* po = part_o + ((size_t)bh * splits * G + r) * D + e;  // chunk s at po[s * G * D]
        int s = grp;
        for (; s + 3 * kGroups < splits; s += 4 * kGroups) {
            float l4[4], v4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                l4[u] = pl[(size_t)(s + u * kGroups) * G];
                v4[u] = po[(size_t)(s + u * kGroups) * G * D];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) acc += __expf(l4[u] - lmax) * v4[u];
        }
        for (; s < splits; s += kGroups) acc += __expf(pl[(size_t)s * G] - lmax) * po[(size_t)s * G * D];
    }
    part[grp][e] = acc;
    __syncthreads();
    if (tid < D) {
        float t = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) t += part[g][tid];
        part[0][tid] = wsum > 0.f ? t / wsum : 0.f;
    }
    __syncthreads();
    if (tid < D / 2) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(o) + (size_t)row * D * 2);
        dst[tid] = pack2<BF16>(part[0][2 * tid], part[0][2 * tid + 1]);
    }
    if (tid == 0) lse[row] = lmax == -INFINITY ? -INFINITY : lmax + logf(wsum);
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
    using L = DecLayout<D>;
    if (a.stage < 0 || a.stage == 0) {
        const int smem_bytes = L::kBytes + 1024;
        auto kern = attn_decode_kernel<D, BF16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        const long n_items = (long)a.groups * a.splits;
        const int grid = (int)(n_items < a.num_sms ? n_items : a.num_sms);
        kern<<<grid, kDecThreads, smem_bytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.seqlens, a.part_o, a.part_l, a.o,
                                                        a.lse, a.Hkv, a.G, a.Nmax, a.splits, a.chunk, (int)n_items,
                                                        a.scale, a.error);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // with one chunk per group the chunk kernel has written O and L itself
    if ((a.stage < 0 || a.stage == 1) && a.splits > 1) {
        const long rows = (long)a.groups * a.G;
        attn_decode_combine_kernel<D, BF16><<<(unsigned)rows, kCombThreads, 0, stream>>>(a.part_o, a.part_l, a.o,
                                                                                         a.lse, a.G, a.splits);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.d == 128) return a.fp16 ? launch_decode_t<128, false>(a, stream) : launch_decode_t<128, true>(a, stream);
    if (a.d == 64) return a.fp16 ? launch_decode_t<64, false>(a, stream) : launch_decode_t<64, true>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
