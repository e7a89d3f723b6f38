// Backward of sparse top-k attention with one shared latent key/value row per key
// (the workload of the cudnn-frontend pull request "Improve performance of SM100 DSA
// backward kernel": keys gathered by top-k index, an attention sink per head, QK width
// 512 or 576 with V = the first 512 columns, per-row top-k lengths, causal or not).
//
// One CTA per (query row i, group of 64 heads).  The query's top-k list is walked in
// tiles of 128 entries, and every product keeps the keys on the TMEM lanes (M = 128):
//   S^T  = K Q^T        [keys x heads]  (K = d_qk, streamed in 64-column chunks)
//   dP^T = V dO^T       [keys x heads]  (the first 512 columns of the same chunks)
//   P^T = exp(S^T - L), dS^T = scale P^T (dP^T - D)        (elementwise warpgroup)
//   dQ^T += K^T dS^T    [d_qk x heads]  (d on the lanes, 128 rows per product)
//   dKV_tile = dS^T Q + [P^T dO, 0]     [keys x d_qk], 64 columns at a time (A = dS^T,
//                                        P^T from TMEM), added to the FP32 accumulator
//                                        with vector reductions of whole 128-byte pieces
// TMEM (512 columns): S^T 0..63 (P^T packed to 16 bits over its first 32 columns),
// dP^T 64..127, dQ^T 128..447 (five 64-column blocks at d_qk = 576, four at 512),
// dKV chunk 448..511; dS^T packed to 16 bits over dP^T's first 32 columns.  Shared memory: Q and dO of the 64 heads (72 + 64 KB), a ring of
// four 16 KB key chunks (128 keys x 64 columns, gathered by eight loader warps with
// cp.async), and dS^T (16 KB).  The key chunks are gathered twice per tile: for S^T /
// dP^T, and again, two at a time, for dQ^T (the whole 128 x 576 tile does not fit
// beside Q and dO).
//
// Roles (512 threads, registers split with setmaxnreg): warps 0-3 elementwise + dKV flush +
// dQ epilogue (thread = TMEM lane = key of the tile, then = d row of dQ^T); warp 4 issues the
// MMAs (whole warp, lane 0 issues); warps 8-15 gather key chunks and, thread 256, load Q / dO.
// More gathering threads keep more copies issued (four loader warps: 14.1 ms, two: 15.5 ms,
// eight: 13.6 ms at H = 128, QK 576, top-k 2048).
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kDsaThreads = 512;
constexpr int kDsaHeads = 64;     // heads per CTA
constexpr int kDsaTile = 128;     // list entries (keys) per tile
constexpr int kDsaDv = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int DQK>
struct DsaLayout {
    static constexpr int kNC = DQK / 64;               // 64-column chunks of a key row
    static constexpr int kNCE = (kNC + 1) & ~1;        // ring entries per pass (even: dQ^T takes pairs)
    static constexpr int kNM = kNCE / 2;               // 128-row dQ^T blocks
    static constexpr int kNV = kDsaDv / 64;            // chunks that also carry V
    static constexpr int kPanel = kDsaHeads * 128;     // 64 rows x 128 bytes
    static constexpr int kChunk = kDsaTile * 128;      // 128 keys x 128 bytes
    static constexpr int kQ = 0;
    static constexpr int kDO = kQ + kNC * kPanel;
    static constexpr int kRing = kDO + kNV * kPanel;
    static constexpr int kDS = kRing + 4 * kChunk;
    // QK = 512: dQ^T needs four TMEM blocks, which leaves 64 columns for P^T and dS^T of a tile
    // and room in shared memory for a separate flush staging buffer, so a tile's dKV products
    // and flush can run under the next tile's gathers (kOvl).
    static constexpr bool kOvl = (DQK == 512);
    static constexpr int kStage = kDS + kChunk;         // kOvl: 16 KB flush staging
    static constexpr int kAux = kStage + (kOvl ? kChunk : 0);
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = 1;      // [4]
    static constexpr int kBarKEmpty = 5;     // [4]
    static constexpr int kBarSFull = 9;
    static constexpr int kBarPReady = 10;
    static constexpr int kBarDkvFull = 11;
    static constexpr int kBarDkvFree = 12;
    static constexpr int kBarDqFull = 13;
    static constexpr int kBarTeardown = 14;
    static constexpr int kBarDqDone = 15;    // the tile's dQ^T products have read dS^T in shared memory
    static constexpr int kBarDkvDone = 16;   // kOvl: the tile's dKV products have read P^T / dS^T
    static constexpr int kNumBars = 17;
    static_assert(kNumBars <= 24, "barrier area");
    static constexpr int kL2eOff = kAux + 8 * 24;       // float [64]: L log2 e
    static constexpr int kDOff = kL2eOff + 4 * 64;      // float [64]: D = dO . O
    static constexpr int kMiscOff = kDOff + 4 * 64;     // tmem base, abort flag
    static constexpr int kBytes = kMiscOff + 64;
    static constexpr uint32_t kTmemS = 0, kTmemDP = 64, kTmemDQ = 128, kTmemDKV = 448;
    // P^T and dS^T (16-bit pairs): over S^T / dP^T, or (kOvl) in the columns after dQ^T
    static constexpr uint32_t kTmemPT = kOvl ? 384 : kTmemS, kTmemDST = kOvl ? 416 : kTmemDP;
    static_assert(kTmemDQ + 64 * kNM <= (kOvl ? kTmemPT : kTmemDKV), "TMEM columns");
    static_assert(kBytes + 1024 <= 232448, "shared memory");
};

struct DsaParams {
    const uint16_t* kv;      // [s_kv, d_qk]
    const uint16_t* o;       // [s_q, H, 512]
    const uint16_t* dout;    // [s_q, H, 512]
    const float* lse;        // [s_q, H]
    const float* sink;       // [H] or nullptr
    const int* idx;          // [s_q, topk]
    const int* topk_len;     // [s_q] or nullptr
    uint16_t* dq;            // [s_q, H, d_qk]
    float* dkv_acc;          // [s_kv, d_qk], zero at launch
    float* dsink;            // [H], zero at launch (nullptr without sinks)
    int s_q, s_kv, H, topk;
    float scale;
    int causal;
    int* error;
};

// Entries of query i's list that take part: position < len_i, 0 <= key < s_kv, and
// key <= i when causal.  Returns the key, or -1.
__device__ __forceinline__ int dsa_key(const DsaParams& p, int i, int len, int e) {
    if (e >= len) return -1;
    const int k = __ldg(p.idx + (size_t)i * p.topk + e);
    if (k < 0 || k >= p.s_kv || (p.causal && k > i)) return -1;
    return k;
}

__device__ __forceinline__ int dsa_len(const DsaParams& p, int i) {
    int len = p.topk;
    if (p.topk_len) len = min(max(__ldg(p.topk_len + i), 0), p.topk);
    return len;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int DQK>
__global__ void __launch_bounds__(kDsaThreads, 1)
dsa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
               const DsaParams p) {
    using L = DsaLayout<DQK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kAux);
    float* l2e_s = reinterpret_cast<float*>(smem + L::kL2eOff);
    float* d_s = reinterpret_cast<float*>(smem + L::kDOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    int* abort_flag = reinterpret_cast<int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int i = blockIdx.x;                    // query row
    const int h0 = blockIdx.y * kDsaHeads;       // first head of the group
    const int len = dsa_len(p, i);
    const int n_tiles = (len + kDsaTile - 1) / kDsaTile;

    if (threadIdx.x == 0) {
        mbar_init(&bars[L::kBarQFull], 1);
        for (int s = 0; s < 4; ++s) {
            mbar_init(&bars[L::kBarKFull + s], 256);
            mbar_init(&bars[L::kBarKEmpty + s], 1);
        }
        mbar_init(&bars[L::kBarSFull], 1);
        mbar_init(&bars[L::kBarPReady], 128);
        mbar_init(&bars[L::kBarDkvFull], 1);
        mbar_init(&bars[L::kBarDkvFree], 128);
        mbar_init(&bars[L::kBarDqFull], 1);
        mbar_init(&bars[L::kBarTeardown], 1);
        mbar_init(&bars[L::kBarDqDone], 1);
        mbar_init(&bars[L::kBarDkvDone], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 4) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard guard{abort_flag, p.error, kWaitLimitNs};

    if (warp < 4) {
        regs_inc<208>();   // 128 x 208 + 128 x 80 + 256 x 96 = 61440 of the 65536 launched
        // ------------------------------------------------ elementwise, dKV flush, dQ epilogue
        const int r = threadIdx.x;                          // TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        // D = dO . O and L log2 e for the 64 heads, and the sink gradient.  Warp w takes heads
        // 16 w .. 16 w + 15, one row at a time: each load instruction covers 512 contiguous bytes.
        {
            const int lane = r & 31;
#pragma unroll 1
            for (int hh = 0; hh < 16; hh += 4) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const size_t row = (size_t)i * p.H + h0 + 16 * warp + hh + q4;
                    const uint4* o4 = reinterpret_cast<const uint4*>(p.o + row * kDsaDv);
                    const uint4* d4 = reinterpret_cast<const uint4*>(p.dout + row * kDsaDv);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 a = __ldg(o4 + 32 * c + lane), b = __ldg(d4 + 32 * c + lane);
                        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
                            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
                            acc[q4] = fmaf(fa.x, fb.x, acc[q4]);
                            acc[q4] = fmaf(fa.y, fb.y, acc[q4]);
                        }
                    }
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[q4] += __shfl_xor_sync(0xffffffffu, acc[q4], o);
                }
                if (lane < 4) {
                    const int h = 16 * warp + hh + lane;
                    const float dsum = lane == 0 ? acc[0] : lane == 1 ? acc[1] : lane == 2 ? acc[2] : acc[3];
                    const float lse = __ldg(p.lse + (size_t)i * p.H + h0 + h);
                    d_s[h] = dsum;
                    l2e_s[h] = lse * kLog2e;
                    if (p.sink != nullptr && p.dsink != nullptr && lse > -INFINITY)
                        atomicAdd(p.dsink + h0 + h, -expf(__ldg(p.sink + h0 + h) - lse) * dsum);
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        const float sl2 = p.scale * kLog2e;
        bool ok = true;
        uint32_t j = 0;  // dKV chunks flushed
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int key = dsa_key(p, i, len, t * kDsaTile + r);
            if (!mbar_wait(&bars[L::kBarSFull], t & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
            // kOvl: the previous tile's dKV products read P^T / dS^T from the columns written below
            if (L::kOvl && t > 0 && !mbar_wait(&bars[L::kBarDkvDone], (t - 1) & 1, guard, kDevTimeoutSoftmax)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // Two halves of 32 heads.  P^T (16-bit pairs) goes over S^T's first 32 columns and
            // dS^T over dP^T's: half 0 writes columns 0-15 of each (heads 0-31, already in
            // registers), half 1 columns 16-31.  dS^T also goes to shared memory for dQ^T.
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t s[32], dp[32];
                tmem_ld32(tmem + lane_base + L::kTmemS + 32 * hf, s);
                tmem_ld32(tmem + lane_base + L::kTmemDP + 32 * hf, dp);
                tmem_wait_ld();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int h = 32 * hf + e;
                    float p0 = 0.f, p1 = 0.f;
                    if (key >= 0) {
                        p0 = ex2_ftz(fmaf(__uint_as_float(s[e]), sl2, -l2e_s[h]));
                        p1 = ex2_ftz(fmaf(__uint_as_float(s[e + 1]), sl2, -l2e_s[h + 1]));
                    }
                    const float g0 = p.scale * p0 * (__uint_as_float(dp[e]) - d_s[h]);
                    const float g1 = p.scale * p1 * (__uint_as_float(dp[e + 1]) - d_s[h + 1]);
                    pk[e >> 1] = bf16x2_bits(p0, p1);
                    dk[e >> 1] = bf16x2_bits(g0, g1);
                }
                tmem_st16(tmem + lane_base + L::kTmemPT + 16 * hf, pk);
                tmem_st16(tmem + lane_base + L::kTmemDST + 16 * hf, dk);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
                    *reinterpret_cast<uint4*>(smem + L::kDS + sw128_offset(r, 4 * hf + c)) = v;
                }
            }
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars[L::kBarPReady]);

            // dKV of this tile, 64 columns at a time, into the FP32 accumulator.  Each warp turns
            // its 32 rows (thread = key) around in shared memory (dS^T's buffer, free once the
            // tile's dQ^T products have read it), so that one reduction instruction covers four
            // whole 128-byte row pieces instead of 32 scattered 16-byte ones.
            if (!L::kOvl && !mbar_wait(&bars[L::kBarDqDone], t & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
            uint8_t* stage = smem + (L::kOvl ? L::kStage : L::kDS) + warp * 4096;     // 32 rows x 128 bytes
            const int lane = r & 31;
            float* rdst[8];   // rows 4 it + lane / 8 of this warp: their accumulator rows + piece offset
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int krow = __shfl_sync(0xffffffffu, key, 4 * it + (lane >> 3));
                rdst[it] = krow >= 0 ? p.dkv_acc + (size_t)krow * DQK + 4 * (lane & 7) : nullptr;
            }
            for (int cc = 0; cc < L::kNC; ++cc, ++j) {
                if (!mbar_wait(&bars[L::kBarDkvFull], j & 1, guard, kDevTimeoutSoftmax)) { ok = false; break; }
                tc_fence_after();
                uint32_t v[2][32];
                tmem_ld32(tmem + lane_base + L::kTmemDKV, v[0]);
                tmem_ld32(tmem + lane_base + L::kTmemDKV + 32, v[1]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars[L::kBarDkvFree]);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                            make_uint4(v[hf][4 * c], v[hf][4 * c + 1], v[hf][4 * c + 2], v[hf][4 * c + 3]);
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int row = 4 * it + (lane >> 3), piece = lane & 7;
                        const float4 f = *reinterpret_cast<const float4*>(stage + row * 128 + ((piece ^ (row & 7)) << 4));
                        if (rdst[it] != nullptr)
                            red_add_v4(rdst[it] + cc * 64 + 32 * hf, f.x, f.y, f.z, f.w);
                    }
                    __syncwarp();
                }
            }
        }
        // dQ epilogue: thread r holds row d = 128 m + r of each dQ^T block (64 heads).
        if (ok) {
            const bool have = n_tiles > 0;
            if (have && !mbar_wait(&bars[L::kBarDqFull], 0, guard, kDevTimeoutSoftmax)) ok = false;
            if (ok) {
                tc_fence_after();
                uint16_t* dq_base = p.dq + ((size_t)i * p.H + h0) * DQK;
                for (int m = 0; m < L::kNM; ++m) {
                    const int d = 128 * m + r;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t v[32];
                        if (have) {
                            tmem_ld32(tmem + lane_base + L::kTmemDQ + 64 * m + 32 * hf, v);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int h = 0; h < 32; ++h) v[h] = 0u;
                        }
                        if (d < DQK) {
#pragma unroll
                            for (int h = 0; h < 32; ++h) {
                                const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[h]));
                                dq_base[(size_t)(32 * hf + h) * DQK + d] = *reinterpret_cast<const uint16_t*>(&b);
                            }
                        }
                    }
                }
            }
        }
    } else if (warp < 8) {
      regs_dec<80>();
      if (warp == 4) {
        // ------------------------------------------------ MMA issuer (the whole warp; lane 0 issues)
        constexpr uint32_t kIdS = idesc_f16(128, 64, true, false, false);    // S^T, dP^T
        constexpr uint32_t kIdQ = idesc_f16(128, 64, true, true, true);      // dQ^T = K^T dS^T
        constexpr uint32_t kIdKV = idesc_f16(128, 64, true, false, true);    // dKV = dS^T Q (+ P^T dO)
        const uint32_t q_base = smem_u32(smem + L::kQ), do_base = smem_u32(smem + L::kDO);
        const uint32_t ring = smem_u32(smem + L::kRing), ds_base = smem_u32(smem + L::kDS);
        bool ok = n_tiles > 0;
        if (ok && !warp_mbar_wait(&bars[L::kBarQFull], 0, guard, kDevTimeoutMma)) ok = false;
        uint32_t k = 0, j = 0;
        // dKV chunk cc = dS^T Q[:, cc] (+ P^T dO[:, cc]), flushed by the elementwise warps
        auto issue_dkv = [&](int cc) -> bool {
            if (!warp_mbar_wait(&bars[L::kBarDkvFree], (j & 1) ^ 1, guard, kDevTimeoutMma)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                warp_mma_ts(tmem + L::kTmemDKV, tmem + L::kTmemDST + 8 * kk,
                            sdesc_sw128(q_base + cc * L::kPanel + kk * 2048, L::kPanel, 1024), kIdKV, kk != 0);
            if (cc < L::kNV) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    warp_mma_ts(tmem + L::kTmemDKV, tmem + L::kTmemPT + 8 * kk,
                                sdesc_sw128(do_base + cc * L::kPanel + kk * 2048, L::kPanel, 1024), kIdKV, 1u);
            }
            warp_mma_commit(&bars[L::kBarDkvFull]);
            ++j;
            return true;
        };
        for (int t = 0; t < n_tiles && ok; ++t) {
            // S^T = K Q^T and dP^T = V dO^T over the key chunks; kOvl: the previous tile's dKV
            // chunks kNC/2 .. kNC-1 interleaved with the first of them
            for (int c = 0; c < L::kNCE; ++c, ++k) {
                const uint32_t slot = k & 3;
                if (!warp_mbar_wait(&bars[L::kBarKFull + slot], (k >> 2) & 1, guard, kDevTimeoutMma)) { ok = false; break; }
                tc_fence_after();
                if (c < L::kNC) {
                    const uint32_t kc = ring + slot * L::kChunk;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(kc + kk * 32, 16, 1024);
                        warp_mma_ss(tmem + L::kTmemS, a, sdesc_sw128(q_base + c * L::kPanel + kk * 32, 16, 1024), kIdS,
                                    (c | kk) != 0);
                        if (c < L::kNV)
                            warp_mma_ss(tmem + L::kTmemDP, a, sdesc_sw128(do_base + c * L::kPanel + kk * 32, 16, 1024),
                                        kIdS, (c | kk) != 0);
                    }
                }
                warp_mma_commit(&bars[L::kBarKEmpty + slot]);
                if (L::kOvl && t > 0 && c < L::kNC / 2 && !issue_dkv(L::kNC / 2 + c)) { ok = false; break; }
            }
            if (!ok) break;
            if (L::kOvl && t > 0) warp_mma_commit(&bars[L::kBarDkvDone]);
            warp_mma_commit(&bars[L::kBarSFull]);
            if (!warp_mbar_wait(&bars[L::kBarPReady], t & 1, guard, kDevTimeoutMma)) { ok = false; break; }
            tc_fence_after();
            // dQ^T += K^T dS^T, two key chunks (128 rows of d) per product
            for (int m = 0; m < L::kNM; ++m, k += 2) {
                const uint32_t slot = k & 3;  // even: the pair is two adjacent slots
                if (!warp_mbar_wait(&bars[L::kBarKFull + slot], (k >> 2) & 1, guard, kDevTimeoutMma) ||
                    !warp_mbar_wait(&bars[L::kBarKFull + slot + 1], ((k + 1) >> 2) & 1, guard, kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kc = ring + slot * L::kChunk;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    warp_mma_ss(tmem + L::kTmemDQ + 64 * m, sdesc_sw128(kc + kk * 2048, L::kChunk, 1024),
                                sdesc_sw128(ds_base + kk * 2048, L::kChunk, 1024), kIdQ, (t | kk) != 0);
                warp_mma_commit(&bars[L::kBarKEmpty + slot]);
                warp_mma_commit(&bars[L::kBarKEmpty + slot + 1]);
                // kOvl: dKV chunk m of this tile between the dQ^T pairs
                if (L::kOvl && !issue_dkv(m)) { ok = false; break; }
            }
            if (!ok) break;
            warp_mma_commit(&bars[L::kBarDqDone]);
            if (!L::kOvl) {
                for (int cc = 0; cc < L::kNC && ok; ++cc)
                    if (!issue_dkv(cc)) ok = false;
            }
        }
        if (L::kOvl && ok && n_tiles > 0) {
            // the last tile's remaining dKV chunks
            for (int cc = L::kNC / 2; cc < L::kNC && ok; ++cc)
                if (!issue_dkv(cc)) ok = false;
            if (ok) warp_mma_commit(&bars[L::kBarDkvDone]);
        }
        if (ok && n_tiles > 0) warp_mma_commit(&bars[L::kBarDqFull]);
        warp_mma_commit(&bars[L::kBarTeardown]);
        mbar_wait_drain(&bars[L::kBarTeardown], 0, kWaitLimitNs);
      }
    } else {
        regs_dec<96>();
        // ------------------------------------------------ gather loaders: eight consecutive threads
        // copy one 128-byte row piece, so a warp's copies cover four whole rows (lines)
        const int r = threadIdx.x - 256;
        const int piece = r & 7, row0 = r >> 3;   // rows row0 + 32 j, j = 0..3
        if (r == 0 && n_tiles > 0) {
            mbar_arrive_expect_tx(&bars[L::kBarQFull], (L::kNC + L::kNV) * L::kPanel);
            const int y = i * p.H + h0;
            for (int c = 0; c < L::kNC; ++c) tma_load_3d(smem + L::kQ + c * L::kPanel, &tm_q, &bars[L::kBarQFull], 64 * c, y, 0);
            for (int c = 0; c < L::kNV; ++c)
                tma_load_3d(smem + L::kDO + c * L::kPanel, &tm_do, &bars[L::kBarQFull], 64 * c, y, 0);
        }
        const uint32_t ring = smem_u32(smem + L::kRing);
        bool ok = true;
        uint32_t k = 0;
        for (int t = 0; t < n_tiles && ok; ++t) {
            uint32_t src_off[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int key = dsa_key(p, i, len, t * kDsaTile + row0 + 32 * jj);
                src_off[jj] = key >= 0 ? ((uint32_t)key * DQK) | 0x80000000u : 0u;
            }
            for (int pass = 0; pass < 2 && ok; ++pass) {
                for (int c = 0; c < L::kNCE; ++c, ++k) {
                    const uint32_t slot = k & 3;
                    if (k >= 4 && !mbar_wait(&bars[L::kBarKEmpty + slot], ((k >> 2) - 1) & 1, guard, kDevTimeoutLoad)) {
                        ok = false;
                        break;
                    }
                    if (c < L::kNC) {
                        const uint32_t dst = ring + slot * L::kChunk;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const uint32_t off = src_off[jj] & 0x7FFFFFFFu;
                            cp_async_16(dst + sw128_offset(row0 + 32 * jj, piece), p.kv + off + 64 * c + 8 * piece,
                                        (src_off[jj] >> 31) ? 16u : 0u);
                        }
                    }
                    cp_async_commit();
                    // Entry k - 2 has landed (two entries stay in flight): publish it.
                    if (k >= 2) {
                        cp_async_wait<2>();
                        fence_proxy_async_smem();
                        mbar_arrive(&bars[L::kBarKFull + ((k - 2) & 3)]);
                    }
                }
            }
        }
        cp_async_wait<0>();
        if (ok) {
            fence_proxy_async_smem();
            for (uint32_t e = (k >= 2 ? k - 2 : 0); e < k; ++e) mbar_arrive(&bars[L::kBarKFull + (e & 3)]);
        }
        if (r == 0 && n_tiles > 0) mbar_wait_drain(&bars[L::kBarQFull], 0, kWaitLimitNs);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dKV (16-bit) from the FP32 accumulator, 4 elements per thread and step.
__global__ void dsa_dkv_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ out, size_t n4) {
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4; e += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[e];
        out[e] = make_uint2(bf16x2_bits(v.x, v.y), bf16x2_bits(v.z, v.w));
    }
}

template <int DQK>
cudaError_t launch_dsa_t(const DsaArgs& a, cudaStream_t stream) {
    using L = DsaLayout<DQK>;
    const int smem_bytes = L::kBytes + 1024;
    auto kern = dsa_bwd_kernel<DQK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    DsaParams p;
    p.kv = static_cast<const uint16_t*>(a.kv);
    p.o = static_cast<const uint16_t*>(a.o);
    p.dout = static_cast<const uint16_t*>(a.dout);
    p.lse = a.lse;
    p.sink = a.sink;
    p.idx = a.idx;
    p.topk_len = a.topk_len;
    p.dq = static_cast<uint16_t*>(a.dq);
    p.dkv_acc = a.dkv_acc;
    p.dsink = a.dsink;
    p.s_q = a.s_q;
    p.s_kv = a.s_kv;
    p.H = a.H;
    p.topk = a.topk;
    p.scale = a.scale;
    p.causal = a.causal;
    p.error = a.error;
    dim3 grid((unsigned)a.s_q, (unsigned)(a.H / kDsaHeads));
    kern<<<grid, kDsaThreads, smem_bytes, stream>>>(a.tm_q, a.tm_do, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dsa_bwd(const DsaArgs& a, cudaStream_t stream) {
    const size_t acc_bytes = (size_t)a.s_kv * a.d_qk * sizeof(float);
    cudaError_t e = cudaMemsetAsync(a.dkv_acc, 0, acc_bytes, stream);
    if (e != cudaSuccess) return e;
    if (a.dsink) {
        e = cudaMemsetAsync(a.dsink, 0, (size_t)a.H * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    e = a.d_qk == 576 ? launch_dsa_t<576>(a, stream) : launch_dsa_t<512>(a, stream);
    if (e != cudaSuccess) return e;
    const size_t n4 = (size_t)a.s_kv * a.d_qk / 4;
    const int grid = (int)((n4 + 255) / 256 < (size_t)a.num_sms * 8 ? (n4 + 255) / 256 : (size_t)a.num_sms * 8);
    dsa_dkv_convert_kernel<<<grid > 0 ? grid : 1, 256, 0, stream>>>(reinterpret_cast<const float4*>(a.dkv_acc),
                                                                     static_cast<uint2*>(a.dkv), n4);
    return cudaGetLastError();
}

}  // namespace gb300
