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
};

// Wait limit for every mbarrier wait in the kernels (nanoseconds of
// %globaltimer).  No single wait in a healthy launch comes near it.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct FwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;   // [BH, N, d], box {64, 128, 1}, 128B swizzle
    void* o;          // [BH, N, d] 16-bit
    float* lse;       // [BH, N]
    int BH, N, d;
    float scale;      // softmax scale applied to QK^T
    int causal;
    int fp16;         // 0 = bf16, 1 = fp16
    int num_sms;
    int* error;       // device error word
};

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    const void* o;    // [BH, N, d]
    const void* dout; // [BH, N, d]
    const float* lse; // [BH, N]
    void* dq;         // [BH, N, d]
    void* dk;
    void* dv;
    float* delta;     // workspace [BH, N]   -D = -rowsum(dO o O)
    float* lse2;      // workspace [BH, N]   -L * log2(e)
    float* dq_acc;    // workspace [BH, N, d] FP32
    int BH, N, d;
    float scale;
    int causal;
    int fp16;
    int num_sms;
    int device;
    int* error;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// stage: -1 = all three kernels; 0 = preprocess; 1 = main kernel; 2 = dQ conversion.
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stage);

}  // namespace gb300
