// attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.  Some callers own every byte of device memory themselves and forbid
// allocations by the libraries they call (a serving engine that carves one
// pre-sized pool at start-up, a host framework that hands plugins only their
// inputs and outputs), or run where cudaMalloc's implicit synchronisation or
// its out-of-memory failure mid-run is not acceptable.  attn_bwd needs a
// caller-provided workspace; this entry point instead uses scratch memory that
// is part of the library image itself: the file-scope device array below.
// The CUDA driver reserves it on a GPU when it loads this file's device code
// (under the default lazy module loading, at the first call's address lookup
// on that GPU; at library load with CUDA_MODULE_LOADING=EAGER) and keeps it
// until the process exits.  It calls no cudaMalloc, cudaFree or other
// allocating routine.
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace gb300 {
namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;

// Scratch shared by every attn_bwd_noalloc call on a device: the D vector,
// L*log2(e) and the FP32 dQ accumulator of the backward pass.  Its contents
// persist from call to call; the backward's first kernel rewrites all of it
// that is read (D, L*log2(e)) and zeroes the dQ accumulator before use.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// symbol is only a host-side stand-in, so the address has to come from
// cudaGetSymbolAddress, once per device, with that device current.
attn_status_t scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace gb300

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                          const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                                          int H, int N, int d, float scale, int causal, attn_dtype_t dtype,
                                          void* stream) {
    const size_t need = attn_bwd_workspace_size(B, H, N, d);
    if (need == 0) {
        // Sizes the backward rejects: let it report the exact reason (it checks sizes before the
        // workspace, and queues nothing).
        return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, B, H, N, d, scale, causal, dtype,
                           stream);
    }
    if (need > gb300::kScratchBytes) {
        // Too large for the fixed array: with no workspace at all the backward refuses with
        // ATTN_ERR_WORKSPACE (or an argument error that takes precedence) and queues nothing.
        return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, B, H, N, d, scale, causal, dtype,
                           stream);
    }
    void* scratch = nullptr;
    const attn_status_t st = gb300::scratch_address(&scratch);
    if (st != ATTN_OK) return st;
    return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, scratch, gb300::kScratchBytes, B, H, N, d, scale, causal,
                       dtype, stream);
}
