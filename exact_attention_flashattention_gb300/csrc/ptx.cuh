// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk),
// tcgen05 (TMEM alloc, MMA, commit, ld/st, fences) and the shared-memory /
// instruction descriptors that tcgen05.mma consumes.  Written from the PTX ISA
// descriptions of these instructions; nothing here is attention-specific.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gb300 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Error words.  A wait that gives up sets the CTA-local abort flag (so the
// other roles stop waiting too) and records `code` in the global error word.
struct WaitGuard {
    volatile int* abort;   // shared memory
    int* error;            // global memory, read back by the host
    uint64_t limit_ns;
};

// Bounded parity wait: true when the phase completed, false on timeout or
// when another role of this CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitGuard& g, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*g.abort) return false;
        if (globaltimer_ns() - t0 > g.limit_ns) {
            *g.abort = 1;
            atomicCAS(g.error, 0, code);
            return false;
        }
    }
}

// Bounded wait with a short sleep between polls, for a thread whose warp should leave issue
// slots to busier warps on the same scheduler.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, const WaitGuard& g, int code) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*g.abort) return false;
        if (globaltimer_ns() - t0 > g.limit_ns) {
            *g.abort = 1;
            atomicCAS(g.error, 0, code);
            return false;
        }
        __nanosleep(256);
    }
}

// The same wait taken by all 32 lanes of a warp, with a warp-uniform outcome
// (a lane that gives up makes the whole warp give up).
__device__ __forceinline__ bool warp_mbar_wait(uint64_t* bar, uint32_t parity, const WaitGuard& g, int code) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, g, code));
}

// Wait that ignores the abort flag (used only at teardown to let in-flight
// asynchronous copies land before shared memory is released); still bounded.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core operand reads, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.mma and tcgen05.commit in warp-uniform form.  The whole warp calls
// them with the same arguments and lane 0 alone issues (the lane test sits
// inside the asm, so the surrounding code stays convergent).  Issuing from a
// region entered by lane 0 only was measured to cap the forward's MMA rate
// well below the tensor pipe's: the per-MMA operand set-up then runs as
// divergent single-thread code.  tcgen05.commit tracks the operations of the
// thread that executes it, so MMAs and their commits all come from lane 0.
//
// D(tmem) = A(smem) * B(smem) (+ D if accumulate)
__device__ __forceinline__ void warp_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D(tmem) = A(tmem) * B(smem) (+ D if accumulate)
__device__ __forceinline__ void warp_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The barrier gets one arrival once every tcgen05 operation lane 0 issued
// before the commit has completed.
__device__ __forceinline__ void warp_mma_commit(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(smem_u32(bar)) : "memory");
}

// One product of several K steps (a chain of tcgen05.mma into the same accumulator) from a
// single asm block: the lane-0 test and the enable-input-d predicates are set once, and every
// later step's shared-memory descriptor is the first one plus a constant added to its low word
// (only the start-address field changes, and it cannot carry out of its 14 bits inside the
// 256 KB shared window).  Offsets are in descriptor units (bytes >> 4).  The per-instruction
// work of the issuing warp is then an add or two and the MMA itself, which matters because the
// MMA warp shares its scheduler with busy elementwise warps.  The first step accumulates when
// acc_first != 0, the later ones always.
#define GB300_MMA_PRE                                                                                  \
    "{\n\t.reg .pred e, p, t;\n\t.reg .b32 l, alo, blo;\n\t.reg .b64 a, b;\n\t"                         \
    "mov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\tsetp.ne.b32 p, %6, 0;\n\tsetp.eq.u32 t, l, l;\n\t"
// SS step: A and B descriptors {lo + off, hi}
#define GB300_MMA_SS_STEP(ao, bo)                                                                      \
    "add.u32 alo, %1, %" #ao ";\n\tadd.u32 blo, %3, %" #bo ";\n\t"                                     \
    "mov.b64 a, {alo, %2};\n\tmov.b64 b, {blo, %4};\n\t"                                               \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, t;\n\t"
// TS step: A in TMEM at %1 + ao (columns), B descriptor {lo + off, hi}
#define GB300_MMA_TS_STEP(ao, bo)                                                                      \
    "add.u32 alo, %1, %" #ao ";\n\tadd.u32 blo, %3, %" #bo ";\n\t"                                     \
    "mov.b64 b, {blo, %4};\n\t"                                                                        \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], b, %5, t;\n\t"

template <int A1, int A2, int A3, int A4, int A5, int A6, int A7, int B1, int B2, int B3, int B4, int B5, int B6,
          int B7>
__device__ __forceinline__ void warp_mma_ss8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t acc_first) {
    asm volatile(GB300_MMA_PRE
                 "mov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t"
                 GB300_MMA_SS_STEP(7, 14) GB300_MMA_SS_STEP(8, 15) GB300_MMA_SS_STEP(9, 16)
                 GB300_MMA_SS_STEP(10, 17) GB300_MMA_SS_STEP(11, 18) GB300_MMA_SS_STEP(12, 19)
                 GB300_MMA_SS_STEP(13, 20) "}"
                 ::"r"(d_tmem), "r"((uint32_t)a_desc), "r"((uint32_t)(a_desc >> 32)), "r"((uint32_t)b_desc),
                 "r"((uint32_t)(b_desc >> 32)), "r"(idesc), "r"(acc_first),
                 "n"(A1), "n"(A2), "n"(A3), "n"(A4), "n"(A5), "n"(A6), "n"(A7),
                 "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7)
                 : "memory");
}
template <int A1, int A2, int A3, int B1, int B2, int B3>
__device__ __forceinline__ void warp_mma_ss4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t acc_first) {
    asm volatile(GB300_MMA_PRE
                 "mov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t"
                 GB300_MMA_SS_STEP(7, 10) GB300_MMA_SS_STEP(8, 11) GB300_MMA_SS_STEP(9, 12) "}"
                 ::"r"(d_tmem), "r"((uint32_t)a_desc), "r"((uint32_t)(a_desc >> 32)), "r"((uint32_t)b_desc),
                 "r"((uint32_t)(b_desc >> 32)), "r"(idesc), "r"(acc_first),
                 "n"(A1), "n"(A2), "n"(A3), "n"(B1), "n"(B2), "n"(B3)
                 : "memory");
}
template <int A1, int A2, int A3, int A4, int A5, int A6, int A7, int B1, int B2, int B3, int B4, int B5, int B6,
          int B7>
__device__ __forceinline__ void warp_mma_ts8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t acc_first) {
    asm volatile(GB300_MMA_PRE
                 "mov.b64 b, {%3, %4};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %5, p;\n\t"
                 GB300_MMA_TS_STEP(7, 14) GB300_MMA_TS_STEP(8, 15) GB300_MMA_TS_STEP(9, 16)
                 GB300_MMA_TS_STEP(10, 17) GB300_MMA_TS_STEP(11, 18) GB300_MMA_TS_STEP(12, 19)
                 GB300_MMA_TS_STEP(13, 20) "}"
                 ::"r"(d_tmem), "r"(a_tmem), "r"(0u), "r"((uint32_t)b_desc), "r"((uint32_t)(b_desc >> 32)),
                 "r"(idesc), "r"(acc_first),
                 "n"(A1), "n"(A2), "n"(A3), "n"(A4), "n"(A5), "n"(A6), "n"(A7),
                 "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7)
                 : "memory");
}
#undef GB300_MMA_PRE
#undef GB300_MMA_SS_STEP
#undef GB300_MMA_TS_STEP

// Descriptor-unit offsets of the K steps of the two operand layouts used here:
//  * K-major SW128, 64-column panels kPanel bytes apart: step kk starts (kk / 4) panels and
//    (kk % 4) x 32 bytes in;
//  * MN-major SW128: step kk starts 16 rows = 2048 bytes further.
// and the TMEM column offsets of a packed 16-bit A operand (8 columns per K step), for the two
// 64-row halves of the key / query index written at columns 0 and 64.
#define GB300_KMAJ_OFFS(panel) 2, 4, 6, (panel) / 16, (panel) / 16 + 2, (panel) / 16 + 4, (panel) / 16 + 6
#define GB300_MNMAJ_OFFS 128, 256, 384, 512, 640, 768, 896
#define GB300_TMEM_A_OFFS 8, 16, 24, 64, 72, 80, 88

// Instruction descriptor, kind::f16 with FP32 accumulation (PTX ISA,
// "Instruction descriptor"): D format bits [4,6), A format [7,10), B format
// [10,13), A major bit 15, B major bit 16 (1 = MN-major), N>>3 at [17,23),
// M>>4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte swizzle layout (PTX ISA,
// "Shared memory descriptor"): start address>>4 at [0,14), leading byte
// offset>>4 at [16,30), stride byte offset>>4 at [32,46), version 1 at
// [46,48), swizzle mode 2 (128B) at [61,64).  Tiles are 1024-byte aligned, so
// the base-offset field stays 0.
//  * K-major SW128 operand (rows of 64 16-bit elements, 8-row atoms of 1 KB):
//    SBO = 1024 (next 8 rows); LBO unused.  Advancing K by 16 elements adds
//    32 bytes to the start address inside the 128-byte row.
//  * MN-major SW128 operand (each 128-byte row holds 64 MN-contiguous elements
//    of one K index): LBO = byte distance between 64-wide MN panels, SBO =
//    1024 (next 8 K rows).  Advancing K by 16 adds 16 rows = 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte
// swizzled panel whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ---- TMEM loads/stores, 32 lanes x 32 bit shape: thread t of the warp gets
// lane (warp quadrant base + t), N consecutive columns.
#define GB300_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
                       "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])
#define GB300_W8(a, o) "r"(a[o + 0]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), \
                       "r"(a[o + 4]), "r"(a[o + 5]), "r"(a[o + 6]), "r"(a[o + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : GB300_R8(r, 0), GB300_R8(r, 8), GB300_R8(r, 16), GB300_R8(r, 24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : GB300_R8(r, 0), GB300_R8(r, 8)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), GB300_W8(r, 0), GB300_W8(r, 8)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), GB300_W8(r, 0), GB300_W8(r, 8), GB300_W8(r, 16), GB300_W8(r, 24)
        : "memory");
}

// ------------------------------------------------------------------ math
// Hardware base-2 exponential (MUFU), flush-to-zero on underflow.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pack two floats into one 32-bit word of 16-bit values, round to nearest even;
// `lo` goes to the low half (the lower K index when used as an MMA operand).
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Packed pairs of FP32 values (Blackwell f32x2 arithmetic).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// Register-count hand-off between warpgroups (must be executed by all warps
// of a warpgroup).
template <int N> __device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N> __device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// 16-byte asynchronous global -> shared copy (cp.async, L2 only); src_bytes 0 writes 16 zero
// bytes and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 256-bit global store (sm_100 and later): eight 32-bit words to a 32-byte aligned address.
__device__ __forceinline__ void st_global_v8(void* gaddr, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(gaddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void red_add_f32(float* gaddr, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gaddr), "f"(a) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* gaddr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 ::"l"(gaddr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

}  // namespace gb300
