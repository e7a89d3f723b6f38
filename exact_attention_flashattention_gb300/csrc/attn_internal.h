// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

// Error codes written by device code into the library's device error word.
enum DeviceError : int {
    kDevOk = 0,
    kDevTimeoutLoad = 1,     // a TMA producer wait gave up
    kDevTimeoutMma = 2,      // the MMA issuer's wait gave up
    kDevTimeoutSoftmax = 3,  // a softmax / elementwise warp's wait gave up
    kDevTimeoutCorr = 4,     // a correction / epilogue warp's wait gave up
    kDevSmemAlign = 5,       // dynamic shared memory could not be 1024-byte aligned (kernel did nothing)
    kDevBadSeqLen = 6,       // packed sequences: offsets decreasing, past the tokens, or longer than the maximum
};

// Wait limit for every mbarrier wait in the kernels (nanoseconds of
// %globaltimer).  No single wait in a healthy launch comes near it.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Row layout of the sequence dimension (see seq.cuh for the addressing).
struct SeqDesc {
    const int* cu;    // device sequence offsets [B + 1], or nullptr when every sequence is N long
    int B, H;
    int N;            // sequence length, or the longest sequence when cu != nullptr
    int token_major;  // 0: [B, H, N, d] (BHSD); 1: [tokens, H, d] (BSHD, or packed when cu != nullptr)
    int tokens;       // rows of a token-major tensor: B N, or cu[B]
    int* error;       // device error word (kDevBadSeqLen)
};

struct FwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;   // 16-bit, box of 64 columns x 128 rows, 128B swizzle
    void* o;          // same layout as q, 16-bit
    float* lse;       // [B, H, N], or [H, tokens] for packed sequences
    SeqDesc seq;
    int BH, N, d;     // BH = B H; N as in seq
    float scale;      // softmax scale applied to QK^T
    int causal;
    int fp16;         // 0 = bf16, 1 = fp16
    int num_sms;
    unsigned int* sched;  // packed sequences: work counter of this launch, zero at launch
    int* error;       // device error word
};

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    const void* o;    // same layout as q
    const void* dout; // same layout as q
    const float* lse; // as FwdArgs::lse
    void* dq;         // same layout as q
    void* dk;
    void* dv;
    // workspace arrays, indexed by the rows of seq_ws_base (seq.cuh); ws_rows rows each
    float* delta;     // -scale D = -scale rowsum(dO o O)
    float* lse2;      // -L log2(e)
    float* dq_acc;    // [ws_rows, d] FP32
    long ws_rows;
    SeqDesc seq;
    unsigned int* sched;  // packed sequences: work counter of the main kernel's launch, zero at launch
    int BH, N, d;
    float scale;
    int causal;
    int fp16;
    int num_sms;
    int device;
    int* error;
};

// Decode: one query row per head against a [B, Hkv, Nmax, d] key/value cache (decode.cu).
struct DecodeArgs {
    CUtensorMap tm_q;        // q [B, Hq, d] viewed as [B Hkv, G, d]; box rows past G are zero-filled
    CUtensorMap tm_k, tm_v;  // caches [B Hkv, Nmax, d]
    const int* seqlens;      // device [B] cache lengths, or nullptr (every batch Nmax)
    float* part_o;           // workspace [B Hkv, splits, G, d]: each chunk's normalised O
    float* part_l;           // workspace [B Hkv, splits, G]: each chunk's L (natural log)
    void* o;                 // [B, Hq, d] 16-bit
    float* lse;              // [B, Hq]
    int groups;              // B Hkv
    int Hkv, G, Nmax, d;
    int splits, chunk;       // key chunks per group, keys per chunk (multiple of 128)
    float scale;
    int fp16;
    int stage;               // -1 both kernels, 0 the chunk kernel, 1 the combination
    int num_sms;
    int* error;
};

// Sparse top-k attention backward with a shared latent key/value row (dsa_bwd.cu).
struct DsaArgs {
    CUtensorMap tm_q;        // q  [s_q H, d_qk] 16-bit, box 64 columns x 64 rows, 128B swizzle
    CUtensorMap tm_do;       // dO [s_q H, 512], same box
    const void* kv;          // [s_kv, d_qk] bf16
    const void* o;           // [s_q, H, 512] bf16
    const void* dout;        // [s_q, H, 512] bf16
    const float* lse;        // [s_q, H]
    const float* sink;       // [H] or nullptr
    const int* idx;          // [s_q, topk]
    const int* topk_len;     // [s_q] or nullptr
    void* dq;                // [s_q, H, d_qk] bf16
    void* dkv;               // [s_kv, d_qk] bf16
    float* dkv_acc;          // [s_kv, d_qk] FP32 workspace
    float* dsink;            // [H] or nullptr
    int s_q, s_kv, H, d_qk, topk;
    float scale;
    int causal;
    int num_sms;
    int* error;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// Zeroes the accumulators, then the main kernel and the dKV conversion (two kernels).
cudaError_t launch_dsa_bwd(const DsaArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
// stage: -1 = all three kernels; 0 = preprocess; 1 = main kernel; 2 = dQ conversion.
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stage);
// The backward's preprocess and dQ conversion kernels (bwd_aux.cu); launch_bwd calls them.
cudaError_t launch_bwd_pre(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_dq_convert(const BwdArgs& a, cudaStream_t stream);

}  // namespace gb300
