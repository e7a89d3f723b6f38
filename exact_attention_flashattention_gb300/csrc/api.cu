// C-ABI entry points of libattn_gb300.so: argument checks, tensor-map
// encoding, workspace carving and kernel dispatch.  Declared in include/attn.h.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace gb300 {

// Device error word written by kernels whose bounded waits gave up.
__device__ int g_device_error = 0;

// Work counters of the persistent kernels' dynamic unit distribution: each launch takes the
// next slot (round robin) and zeroes it on its stream before the kernel runs, so launches in
// flight at the same time (other streams, or graph replays) use different counters as long as
// fewer than kSchedSlots of them overlap.
constexpr int kSchedSlots = 1024;
__device__ unsigned int g_sched_counters[kSchedSlots];

namespace {

thread_local int t_last_launches = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct DevInfo {
    int device = 0;
    int sms = 0;
    int* err_ptr = nullptr;
    unsigned int* sched_base = nullptr;
};

// Per-device cache of the SM count and of the device address of the error word.
bool dev_info(DevInfo& out) {
    static std::mutex mu;
    static DevInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
        DevInfo di;
        di.device = dev;
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err_ptr), g_device_error) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&di.sched_base), g_sched_counters) != cudaSuccess)
            return false;
        cache[dev] = di;
        have[dev] = true;
    }
    out = cache[dev];
    return true;
}

// [BH, N, d] 16-bit tensor, box {64, 128, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [tokens, H, d] 16-bit tensor (BSHD, or packed sequences), box {64, 1, 128}: the same
// 128 rows x 128 bytes in shared memory as the heads-major box.
bool make_map_tokens(CUtensorMap* m, const void* base, int H, int tokens, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_seq(CUtensorMap* m, const void* base, const SeqDesc& s, int d) {
    return s.token_major ? make_map_tokens(m, base, s.H, s.tokens, d) : make_map(m, base, s.B * s.H, s.N, d);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [rows, width] 16-bit row array viewed as {width, rows, 1}, box {64, box_rows, 1}.
bool make_map_rows(CUtensorMap* m, const void* base, int rows, int width, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)rows * width * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A zeroed work counter for one launch on `stream` (nullptr if the memset could not be queued).
unsigned int* take_sched_counter(const DevInfo& di, cudaStream_t stream) {
    static std::atomic<unsigned int> next{0};
    unsigned int* p = di.sched_base + (next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
    if (cudaMemsetAsync(p, 0, sizeof(unsigned int), stream) != cudaSuccess) return nullptr;
    return p;
}

size_t n_pad_of(int N) { return ((size_t)N + 127) / 128 * 128; }

// Rows of each backward workspace array: B H blocks of N_pad rows, or for packed sequences
// H blocks of 128 (ceil(tokens / 128) + B) rows (seq_ws_base in seq.cuh).
size_t ws_rows(const SeqDesc& s) {
    return s.cu != nullptr ? (size_t)s.H * 128 * (((size_t)s.tokens + 127) / 128 + (size_t)s.B)
                           : (size_t)s.B * s.H * n_pad_of(s.N);
}

// Checks the sizes and layout arguments and fills the sequence descriptor (error word unset).
attn_status_t check_seq(int B, int H, int N, int d, attn_layout_t layout, const int* cu_seqlens, int total_tokens,
                        SeqDesc& s) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (layout != ATTN_LAYOUT_BHSD && layout != ATTN_LAYOUT_BSHD && layout != ATTN_LAYOUT_PACKED)
        return ATTN_ERR_INVALID_ARG;
    const bool packed = layout == ATTN_LAYOUT_PACKED;
    if (packed != (cu_seqlens != nullptr)) return ATTN_ERR_INVALID_ARG;
    if (packed && total_tokens < 0) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (packed && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return ATTN_ERR_ALIGNMENT;
    s.cu = cu_seqlens;
    s.B = B;
    s.H = H;
    s.N = N;
    s.token_major = layout != ATTN_LAYOUT_BHSD;
    s.tokens = packed ? total_tokens : 0;
    s.error = nullptr;
    if (layout == ATTN_LAYOUT_BSHD) {
        if ((long long)B * N >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
        s.tokens = B * N;
    }
    if ((long long)ws_rows(s) * d >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// The fixed-length layout's checks (existing entry points).
attn_status_t check_sizes(int B, int H, int N, int d) {
    SeqDesc s;
    return check_seq(B, H, N, d, ATTN_LAYOUT_BHSD, nullptr, 0, s);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t delta, lse2, dq_acc, total;
};
WsLayout ws_layout(const SeqDesc& s, int d) {
    WsLayout w;
    // whole 128-row tiles of every sequence fit, so the kernels always move full tiles
    const size_t rows = ws_rows(s);
    w.delta = 0;
    w.lse2 = align_up(w.delta + rows * 4, 256);
    w.dq_acc = align_up(w.lse2 + rows * 4, 256);
    w.total = align_up(w.dq_acc + rows * (size_t)d * 4, 256);
    return w;
}
WsLayout ws_layout(int B, int H, int N, int d) {
    SeqDesc s;
    check_seq(B, H, N, d, ATTN_LAYOUT_BHSD, nullptr, 0, s);
    return ws_layout(s, d);
}

// Decode work split.  The finest split, chunks of 512 KB of K / V (1024 keys at d = 128, 2048 at
// d = 64: eight or sixteen 128-key tiles), sizes the workspace and is a function of the sizes
// only, so the workspace size needs no device.
void decode_plan(int Nmax, int d, int& splits, int& chunk) {
    chunk = d == 128 ? 1024 : 2048;
    splits = (Nmax + chunk - 1) / chunk;
}

// The split a launch uses: chunks of c >= that many tiles, c chosen so that the persistent grid's
// waves times an item's length (c tiles plus one tile's worth of per-item cost: the first S and
// the epilogue) is smallest, i.e. the items fill the SMs evenly.  Never finer than the workspace's
// split.  GQA B=1 Hkv=8 N=131072 d=128 on 152 SMs: 152 chunks of 54 tiles instead of 1024 of 8.
void decode_plan_launch(int groups, int Nmax, int d, int sms, int& splits, int& chunk) {
    const int base = d == 128 ? 8 : 16;
    const long tiles = (Nmax + 127) / 128;
    long best_c = base, best_cost = -1;
    for (long c = base;; ++c) {
        const long items = (long)groups * ((tiles + c - 1) / c);
        const long waves = (items + sms - 1) / sms;
        const long cost = waves * (c + 1);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_c = c;
        }
        if (c >= tiles) break;
    }
    chunk = (int)(best_c * 128);
    splits = (int)((tiles + best_c - 1) / best_c);
}

attn_status_t check_decode(int B, int Hq, int Hkv, int Nmax, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nmax <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (Hq / Hkv > 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * Hkv * Nmax * d >= (1ll << 31) || (long long)B * Hq * d >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

struct DecodeWs {
    size_t part_l, total;
};
DecodeWs decode_ws(int B, int Hq, int Hkv, int Nmax, int d) {
    int splits, chunk;
    decode_plan(Nmax, d, splits, chunk);
    const size_t rows = (size_t)B * Hkv * splits * (Hq / Hkv);
    DecodeWs w;
    w.part_l = align_up(rows * d * 4, 256);
    w.total = align_up(w.part_l + rows * 4, 256);
    return w;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" {

attn_status_t attn_fwd_layout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int max_seqlen, int d, float scale, int causal, attn_dtype_t dtype,
                              attn_layout_t layout, const int* cu_seqlens, int total_tokens, void* stream) {
    t_last_launches = 0;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_INVALID_ARG;
    SeqDesc seq;
    attn_status_t st = check_seq(B, H, max_seqlen, d, layout, cu_seqlens, total_tokens, seq);
    if (st != ATTN_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_ALIGNMENT;
    if (seq.token_major && seq.tokens == 0) return ATTN_OK;  // packed, every sequence empty: nothing to do
    DevInfo di;
    if (!dev_info(di)) return ATTN_ERR_CUDA;
    seq.error = di.err_ptr;
    FwdArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!make_map_seq(&a.tm_q, q, seq, d) || !make_map_seq(&a.tm_k, k, seq, d) || !make_map_seq(&a.tm_v, v, seq, d))
        return ATTN_ERR_CUDA;
    a.o = o;
    a.lse = lse;
    a.seq = seq;
    a.BH = B * H;
    a.N = max_seqlen;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.fp16 = dtype == ATTN_FP16;
    a.num_sms = di.sms;
    a.error = di.err_ptr;
    a.sched = nullptr;
    if (a.seq.cu) {  // packed sequences: dynamic distribution
        a.sched = take_sched_counter(di, static_cast<cudaStream_t>(stream));
        if (!a.sched) return ATTN_ERR_CUDA;
    }
    if (launch_fwd(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_launches = 1;
    return ATTN_OK;
}

attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                          int d, float scale, int causal, attn_dtype_t dtype, void* stream) {
    return attn_fwd_layout(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, ATTN_LAYOUT_BHSD, nullptr, 0, stream);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                       float scale, int causal, void* stream) {
    return attn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, ATTN_BF16, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
    if (check_sizes(B, H, N, d) != ATTN_OK) return 0;
    return ws_layout(B, H, N, d).total;
}

size_t attn_bwd_layout_workspace_size(int B, int H, int max_seqlen, int d, attn_layout_t layout,
                                      int total_tokens) {
    // the offsets themselves are not needed for the size; a dummy non-null pointer selects packed
    static const int kDummy = 0;
    SeqDesc s;
    if (check_seq(B, H, max_seqlen, d, layout, layout == ATTN_LAYOUT_PACKED ? &kDummy : nullptr, total_tokens, s) !=
        ATTN_OK)
        return 0;
    return ws_layout(s, d).total;
}

}  // extern "C"

namespace {
attn_status_t bwd_common(int stage, const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                         int B, int H, int N, int d, float scale, int causal, attn_dtype_t dtype,
                         attn_layout_t layout, const int* cu_seqlens, int total_tokens, void* stream) {
    t_last_launches = 0;
    if (stage < -1 || stage > 2) return ATTN_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_INVALID_ARG;
    SeqDesc seq;
    attn_status_t st = check_seq(B, H, N, d, layout, cu_seqlens, total_tokens, seq);
    if (st != ATTN_OK) return st;
    const WsLayout w = ws_layout(seq, d);
    if (!workspace || workspace_bytes < w.total) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGNMENT;
    const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv};
    for (const void* p : ptrs)
        if (!aligned16(p)) return ATTN_ERR_ALIGNMENT;
    if (seq.token_major && seq.tokens == 0) return ATTN_OK;  // packed, every sequence empty: nothing to do
    DevInfo di;
    if (!dev_info(di)) return ATTN_ERR_CUDA;
    seq.error = di.err_ptr;
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    const int BH = B * H;
    if (!make_map_seq(&a.tm_q, q, seq, d) || !make_map_seq(&a.tm_k, k, seq, d) || !make_map_seq(&a.tm_v, v, seq, d) ||
        !make_map_seq(&a.tm_do, dout, seq, d))
        return ATTN_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.delta = reinterpret_cast<float*>(ws + w.delta);
    a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    a.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
    a.ws_rows = (long)ws_rows(seq);
    a.seq = seq;
    a.BH = BH;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.fp16 = dtype == ATTN_FP16;
    a.num_sms = di.sms;
    a.device = di.device;
    a.error = di.err_ptr;
    a.sched = nullptr;
    if (seq.cu && (stage < 0 || stage == 1)) {  // packed sequences: dynamic distribution
        a.sched = take_sched_counter(di, static_cast<cudaStream_t>(stream));
        if (!a.sched) return ATTN_ERR_CUDA;
    }
    if (launch_bwd(a, static_cast<cudaStream_t>(stream), stage) != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_launches = stage < 0 ? 3 : 1;
    return ATTN_OK;
}
}  // namespace

extern "C" {

attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          int B, int H, int N, int d, float scale, int causal, attn_dtype_t dtype, void* stream) {
    return bwd_common(-1, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
                      dtype, ATTN_LAYOUT_BHSD, nullptr, 0, stream);
}

attn_status_t attn_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                             size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                             attn_dtype_t dtype, void* stream) {
    if (stage < 0 || stage > 2) {
        t_last_launches = 0;
        return ATTN_ERR_INVALID_ARG;
    }
    return bwd_common(stage, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale,
                      causal, dtype, ATTN_LAYOUT_BHSD, nullptr, 0, stream);
}

attn_status_t attn_bwd_layout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, int B, int H, int max_seqlen, int d, float scale, int causal,
                              attn_dtype_t dtype, attn_layout_t layout, const int* cu_seqlens, int total_tokens,
                              void* stream) {
    return bwd_common(-1, q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, max_seqlen, d, scale,
                      causal, dtype, layout, cu_seqlens, total_tokens, stream);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                       int H, int N, int d, float scale, int causal, void* stream) {
    return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, d, scale, causal,
                       ATTN_BF16, stream);
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nmax, int d) {
    if (check_decode(B, Hq, Hkv, Nmax, d) != ATTN_OK) return 0;
    return decode_ws(B, Hq, Hkv, Nmax, d).total;
}

attn_status_t attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                          const int* cache_seqlens, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                          int Nmax, int d, float scale, attn_dtype_t dtype, void* stream) {
    t_last_launches = 0;
    if (!q || !k_cache || !v_cache || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_decode(B, Hq, Hkv, Nmax, d);
    if (st != ATTN_OK) return st;
    const DecodeWs w = decode_ws(B, Hq, Hkv, Nmax, d);
    if (!workspace || workspace_bytes < w.total) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGNMENT;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_ALIGNMENT;
    if (cache_seqlens && (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u) != 0) return ATTN_ERR_ALIGNMENT;
    DevInfo di;
    if (!dev_info(di)) return ATTN_ERR_CUDA;
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    const int G = Hq / Hkv;
    if (!make_map(&a.tm_q, q, B * Hkv, G, d) || !make_map(&a.tm_k, k_cache, B * Hkv, Nmax, d) ||
        !make_map(&a.tm_v, v_cache, B * Hkv, Nmax, d))
        return ATTN_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.seqlens = cache_seqlens;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_l = reinterpret_cast<float*>(ws + w.part_l);
    a.o = o;
    a.lse = lse;
    a.groups = B * Hkv;
    a.Hkv = Hkv;
    a.G = G;
    a.Nmax = Nmax;
    a.d = d;
    decode_plan_launch(B * Hkv, Nmax, d, di.sms, a.splits, a.chunk);
    a.scale = scale;
    a.fp16 = dtype == ATTN_FP16;
    a.stage = -1;
    a.num_sms = di.sms;
    a.error = di.err_ptr;
    if (launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_launches = a.splits > 1 ? 2 : 1;
    return ATTN_OK;
}

size_t attn_dsa_bwd_workspace_size(int s_kv, int d_qk) {
    if (s_kv <= 0 || (d_qk != 512 && d_qk != 576)) return 0;
    return align_up((size_t)s_kv * d_qk * sizeof(float), 256);
}

attn_status_t attn_dsa_bwd(const void* q, const void* kv, const void* o, const void* dout, const float* lse,
                           const float* sink, const int* topk_idx, const int* topk_len, void* dq, void* dkv,
                           float* dsink, void* workspace, size_t workspace_bytes, int s_q, int s_kv, int H, int d_qk,
                           int d_v, int topk, float scale, int causal, void* stream) {
    t_last_launches = 0;
    if (!q || !kv || !o || !dout || !lse || !topk_idx || !dq || !dkv) return ATTN_ERR_INVALID_ARG;
    if (sink && !dsink) return ATTN_ERR_INVALID_ARG;
    if (s_q <= 0 || s_kv <= 0 || H <= 0 || topk <= 0) return ATTN_ERR_INVALID_ARG;
    if (H % 64 != 0 || (d_qk != 512 && d_qk != 576) || d_v != 512) return ATTN_ERR_UNSUPPORTED;
    if ((long long)s_q * H * d_qk >= (1ll << 31) || (long long)s_kv * d_qk >= (1ll << 31) ||
        (long long)s_q * topk >= (1ll << 31))
        return ATTN_ERR_UNSUPPORTED;
    const size_t need = attn_dsa_bwd_workspace_size(s_kv, d_qk);
    if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGNMENT;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dkv))
        return ATTN_ERR_ALIGNMENT;
    auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (!a4(lse) || !a4(topk_idx) || (sink && !a4(sink)) || (sink && !a4(dsink)) || (topk_len && !a4(topk_len)))
        return ATTN_ERR_ALIGNMENT;
    DevInfo di;
    if (!dev_info(di)) return ATTN_ERR_CUDA;
    DsaArgs a;
    std::memset(&a, 0, sizeof(a));
    // q and dO as 2-D row arrays [s_q H, width]; one box = 64 heads x 64 columns.
    if (!make_map_rows(&a.tm_q, q, s_q * H, d_qk, 64) || !make_map_rows(&a.tm_do, dout, s_q * H, d_v, 64))
        return ATTN_ERR_CUDA;
    a.kv = kv;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.sink = sink;
    a.idx = topk_idx;
    a.topk_len = topk_len;
    a.dq = dq;
    a.dkv = dkv;
    a.dkv_acc = static_cast<float*>(workspace);
    a.dsink = sink ? dsink : nullptr;
    a.s_q = s_q;
    a.s_kv = s_kv;
    a.H = H;
    a.d_qk = d_qk;
    a.topk = topk;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.num_sms = di.sms;
    a.error = di.err_ptr;
    if (launch_dsa_bwd(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_launches = 2;
    return ATTN_OK;
}

const char* attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG:
            return "ATTN_ERR_INVALID_ARG: null pointer, non-positive size, bad dtype or layout, or (device) "
                   "inconsistent sequence offsets";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: d must be 64 or 128 and B*H*N*d below 2^31";
        case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT: pointers must be 16-byte aligned (workspace 256)";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel wait gave up; outputs are incomplete";
    }
    return "unknown attn_status_t";
}

attn_status_t attn_last_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
        if (v == kDevSmemAlign) return ATTN_ERR_CUDA;
        if (v == kDevBadSeqLen) return ATTN_ERR_INVALID_ARG;
        return ATTN_ERR_TIMEOUT;
    }
    return ATTN_OK;
}

int attn_last_launch_count(void) { return t_last_launches; }

}  // extern "C"
