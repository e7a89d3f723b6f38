/*
 * attn.h - C ABI of the GB300 (sm_103a) fused exact-attention library
 * (libattn_gb300.so).
 *
 * The operations are those of "Writing Speed-of-Light Attention Backward
 * Kernel for 5090 in CUDA", section "Mathematical Formulation":
 *
 *   forward   S = scale * Q K^T + M,  L_i = log sum_j exp(S_ij),
 *             P = exp(S - L),  O = P V
 *   backward  D = rowsum(dO o O),  dV = P^T dO,  dP = dO V^T,
 *             dS = P o (dP - D 1^T),  dQ = scale * dS K,  dK = scale * dS^T Q
 *
 * where M_ij = -inf for key j > query i when `causal` is non-zero (the
 * diagonal is kept) and 0 otherwise.  The page writes 1/sqrt(d) for the
 * scale; here it is the caller's `scale`.  S and P are never written to
 * global memory: the backward recomputes P from the saved L.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers, owned by the caller, allocated
 *    on the current CUDA device.  The library allocates no device memory.
 *  - Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d] arrays of 16-bit
 *    floats (bfloat16, or float16 for the *_ex calls with ATTN_FP16), row
 *    d fastest.  L (lse) is a contiguous FP32 [B, H, N] array, natural log.
 *  - Supported sizes: d in {64, 128}; any N >= 1 (a last tile of fewer than
 *    128 rows is handled with zero-filled loads and masking); B, H >= 1;
 *    B*H*N_pad*d < 2^31 with N_pad = 128 ceil(N / 128).  Every pointer must be
 *    16-byte aligned.  Anything else returns an error code before any work is
 *    queued.
 *  - Outputs are overwritten, never accumulated.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream).  A status of ATTN_OK means the work was queued.  Launch
 *    failures are reported as ATTN_ERR_CUDA.  A kernel whose internal wait
 *    gave up (it never should) records that in a device error word, which
 *    attn_last_device_error() reads back.
 *  - No C++ exception crosses this interface.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad dtype   */
    ATTN_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, or too large             */
    ATTN_ERR_ALIGNMENT = 3,    /* a pointer not 16-byte aligned                */
    ATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than required      */
    ATTN_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed             */
    ATTN_ERR_TIMEOUT = 6       /* a kernel-internal wait gave up (device word) */
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype_t;

/*
 * Memory layout of Q, K, V, O, dO, dQ, dK, dV and L for the *_layout calls.
 * The pages' kernels use [B, H, N, d] (ATTN_LAYOUT_BHSD, the layout of every
 * call without "_layout").  "Dense B200 attention from scratch"
 * (b200-attention, Appendix "Benchmark Calibration") also ships a direct-BSHD
 * variant; the flash_attention_cuda README lists variable-length sequence
 * packing among the features it leaves out.
 *   ATTN_LAYOUT_BHSD    tensors [B, H, N, d];  L [B, H, N]
 *   ATTN_LAYOUT_BSHD    tensors [B, N, H, d];  L [B, H, N]
 *   ATTN_LAYOUT_PACKED  tensors [total_tokens, H, d] holding B sequences back
 *                       to back: sequence b is rows cu_seqlens[b] ..
 *                       cu_seqlens[b+1] - 1 (lengths may differ, may be 0);
 *                       L [H, total_tokens].  Attention never crosses a
 *                       sequence boundary; the causal mask is per sequence.
 */
typedef enum { ATTN_LAYOUT_BHSD = 0, ATTN_LAYOUT_BSHD = 1, ATTN_LAYOUT_PACKED = 2 } attn_layout_t;

/*
 * Forward pass (the page's forward equations, section "Mathematical
 * Formulation").  Reads q, k, v [B,H,N,d]; writes o [B,H,N,d] and
 * lse [B,H,N] (L, natural log, FP32), which attn_bwd needs.  BF16 data.
 */
ATTN_API attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int H, int N, int d, float scale, int causal, void *stream);

/* attn_fwd with an explicit 16-bit element type (ATTN_BF16 or ATTN_FP16). */
ATTN_API attn_status_t attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int H, int N, int d, float scale, int causal,
                          attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_ex for the layouts of attn_layout_t.  `max_seqlen` is N for the
 * fixed-length layouts and, for ATTN_LAYOUT_PACKED, an upper bound on every
 * sequence length (the work is laid out for it; a tight bound wastes least).
 * `cu_seqlens` is NULL except for ATTN_LAYOUT_PACKED, where it is a DEVICE
 * array of B + 1 int32 offsets, 4-byte aligned, non-decreasing, from 0 to
 * `total_tokens` (the host does not read it; `total_tokens` is ignored for the
 * other layouts).  Offsets that break these rules are detected on the device:
 * the offending sequences are skipped (their outputs are not written) and
 * attn_last_device_error() returns ATTN_ERR_INVALID_ARG.  With
 * total_tokens == 0 nothing is queued.  For ATTN_LAYOUT_PACKED the call also
 * queues, before the kernel, a 4-byte memset of one of the library's 1024
 * per-launch work counters (taken round robin), so at most 1024 packed
 * forwards may be in flight at once across all streams of a device.
 */
ATTN_API attn_status_t attn_fwd_layout(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int max_seqlen, int d, float scale, int causal,
                              attn_dtype_t dtype, attn_layout_t layout, const int *cu_seqlens,
                              int total_tokens, void *stream);

/*
 * Bytes of device workspace attn_bwd needs: the D vector and L*log2(e)
 * (FP32 [B,H,N_pad] each) and the FP32 dQ accumulator [B,H,N_pad,d], with
 * N_pad = 128 ceil(N / 128).  Returns 0 for sizes attn_bwd would reject.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass (the page's backward equations, section "Mathematical
 * Formulation", with the tiling of its pseudocode: parallel over key/value
 * tiles, dQ partials combined in FP32).  Reads q, k, v, o, dout [B,H,N,d]
 * and lse [B,H,N] as written by attn_fwd for the same q, k, v, scale and
 * causal; writes dq, dk, dv [B,H,N,d].  `workspace` is caller-owned device
 * memory of at least attn_bwd_workspace_size() bytes, 256-byte aligned; its
 * contents on entry do not matter and are clobbered.
 */
ATTN_API attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const void *dout, const float *lse, void *dq, void *dk, void *dv,
                       void *workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, int causal, void *stream);

/* attn_bwd with an explicit 16-bit element type. */
ATTN_API attn_status_t attn_bwd_ex(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, void *dq, void *dk, void *dv,
                          void *workspace, size_t workspace_bytes, int B, int H, int N, int d,
                          float scale, int causal, attn_dtype_t dtype, void *stream);

/*
 * Workspace bytes for attn_bwd_layout: three row-indexed arrays as for
 * attn_bwd_workspace_size, with B H N_pad rows (fixed-length layouts) or
 * H 128 (ceil(total_tokens / 128) + B) rows (packed: every sequence's rows
 * start on a 128-row boundary).  0 for arguments it would reject.
 */
ATTN_API size_t attn_bwd_layout_workspace_size(int B, int H, int max_seqlen, int d, attn_layout_t layout,
                                               int total_tokens);

/*
 * attn_bwd_ex for the layouts of attn_layout_t; the layout arguments as for
 * attn_fwd_layout, and lse as that call wrote it.
 */
ATTN_API attn_status_t attn_bwd_layout(const void *q, const void *k, const void *v, const void *o,
                              const void *dout, const float *lse, void *dq, void *dk, void *dv,
                              void *workspace, size_t workspace_bytes, int B, int H, int max_seqlen,
                              int d, float scale, int causal, attn_dtype_t dtype, attn_layout_t layout,
                              const int *cu_seqlens, int total_tokens, void *stream);

/*
 * The three kernels attn_bwd_ex queues, one at a time, for callers that time
 * them separately or interleave other work on the stream.  stage 0: the
 * preprocess (D = rowsum(dO o O), L log2(e), zeroing the FP32 dQ
 * accumulator); stage 1: the main kernel (dK, dV, and the dQ partials added
 * into the accumulator); stage 2: conversion of the accumulator to dq.
 * Arguments as attn_bwd_ex; the workspace must persist across the three
 * calls.  Queuing stages 0, 1, 2 in that order on one stream is exactly one
 * attn_bwd_ex call.  Any other stage value returns ATTN_ERR_INVALID_ARG.
 */
ATTN_API attn_status_t attn_bwd_stage(int stage, const void *q, const void *k, const void *v,
                             const void *o, const void *dout, const float *lse, void *dq, void *dk,
                             void *dv, void *workspace, size_t workspace_bytes, int B, int H, int N,
                             int d, float scale, int causal, attn_dtype_t dtype, void *stream);

/*
 * Size of the fixed scratch array that attn_bwd_noalloc uses (64 MiB).
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Backward pass for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for callers that own all
 * device memory themselves and forbid allocations by the code they call (a
 * serving engine with one pool sized at start-up, a plugin host that hands out
 * only inputs and outputs), or that cannot accept cudaMalloc's implicit
 * synchronisation or a late out-of-memory failure.
 *
 * Same computation and arguments as attn_bwd_ex, minus the workspace: the
 * scratch it needs (attn_bwd_workspace_size(B, H, N, d) bytes) comes from one
 * fixed device array of ATTN_NOALLOC_SCRATCH_BYTES inside this library.  The
 * driver reserves that array on a GPU when it loads the device code that holds
 * it: under CUDA's default lazy module loading that is the first
 * attn_bwd_noalloc call on that GPU (which resolves the array's address), and
 * the library load itself only with CUDA_MODULE_LOADING=EAGER.  That first
 * call can therefore fail with ATTN_ERR_CUDA if the GPU has less than
 * ATTN_NOALLOC_SCRATCH_BYTES free; a caller that needs the reservation up
 * front makes one call at start-up.  The array then stays reserved until the
 * process exits, and no call allocates or frees memory.
 *  - Sizes whose scratch exceeds ATTN_NOALLOC_SCRATCH_BYTES return
 *    ATTN_ERR_WORKSPACE and queue nothing; other argument errors are those of
 *    attn_bwd_ex.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents (the backward rewrites or zeroes all of it that it reads).
 *    Calls whose work overlaps on the GPU (different streams without ordering
 *    between them) race on the array: order them.
 */
ATTN_API attn_status_t attn_bwd_noalloc(const void *q, const void *k, const void *v,
                               const void *o, const void *dout, const float *lse, void *dq,
                               void *dk, void *dv, int B, int H, int N, int d, float scale,
                               int causal, attn_dtype_t dtype, void *stream);

/*
 * Decode: attention of one new query per head against a key/value cache (the
 * forward equations with a single query row and no mask; the
 * flash_attention_cuda README leaves this "different, memory-bound problem"
 * out).  For batch b and query head h, with G = Hq / Hkv query heads sharing
 * KV head h / G (grouped-query attention; G = 1 is plain multi-head):
 *   o[b, h, :] = softmax(scale q[b, h, :] K_b^T) V_b,
 *   lse[b, h]  = log sum_j exp(scale q[b, h, :] . K_b[j, :])
 * over the cached keys j < len_b of K_b = k_cache[b, h / G], V_b likewise.
 *   q, o        [B, Hq, d] 16-bit;  lse [B, Hq] FP32 (natural log)
 *   k_cache,
 *   v_cache     [B, Hkv, Nmax, d] 16-bit
 *   cache_seqlens  NULL (every len_b = Nmax) or a DEVICE int32 array [B],
 *               4-byte aligned, each 0 <= len_b <= Nmax.  A length outside
 *               that range is treated as 0 and attn_last_device_error()
 *               returns ATTN_ERR_INVALID_ARG; len_b = 0 gives o = 0 and
 *               lse = -inf.
 * Requires Hq a multiple of Hkv, G <= 128, d in {64, 128}, the sizes of the
 * other calls' limits, and a caller-owned `workspace` of at least
 * attn_decode_workspace_size() bytes, 256-byte aligned (the keys are split
 * into chunks processed in parallel; the workspace holds each chunk's partial
 * result).  Queues two kernels: the chunk kernel and their combination, or
 * the chunk kernel alone when the launch takes one chunk per (batch, KV head)
 * (it then writes o and lse itself; attn_last_launch_count() says which).
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nmax, int d);
ATTN_API attn_status_t attn_decode(const void *q, const void *k_cache, const void *v_cache, void *o,
                          float *lse, const int *cache_seqlens, void *workspace,
                          size_t workspace_bytes, int B, int Hq, int Hkv, int Nmax, int d,
                          float scale, attn_dtype_t dtype, void *stream);

/*
 * Backward of sparse top-k attention with one shared latent key/value row per
 * key, the workload of "Improve performance of SM100 DSA backward kernel"
 * (cudnn-frontend pull request 684, PR description): every head of query row i
 * attends to the keys its top-k list names, gathered from one latent row per
 * key; K is the whole row (d_qk = 512 or 576 columns) and V its first d_v = 512
 * columns; an optional per-head sink logit joins each softmax with no value
 * row.  With e the valid entries of row i's list (position e < len_i, where
 * len_i = min(topk_len[i], topk) or topk if topk_len is NULL;
 * 0 <= topk_idx[i, e] < s_kv; and topk_idx[i, e] <= i when causal), and the
 * forward's O and L (L including the sink), the call computes, as in the dense
 * backward ("Writing Speed-of-Light Attention Backward Kernel for 5090 in
 * CUDA", "Mathematical Formulation"):
 *   D = dO . O,  P_e = exp(scale q . k_e - L),  dS_e = P_e (dO . v_e - D)
 *   dq   = scale sum_e dS_e k_e
 *   dkv[topk_idx[i, e]] += scale dS_e q (all d_qk columns) + P_e dO (first 512)
 *   dsink_h = - sum_i exp(sink_h - L_ih) D_ih
 * A key listed twice in a row counts twice.  Rows with no valid entry get dq = 0.
 *
 * Layouts (all DEVICE pointers, caller-owned, bf16 unless noted):
 *   q [s_q, H, d_qk], kv [s_kv, d_qk], o and dout [s_q, H, 512],
 *   lse FP32 [s_q, H] (natural log), sink FP32 [H] or NULL,
 *   topk_idx int32 [s_q, topk], topk_len int32 [s_q] or NULL;
 *   outputs dq [s_q, H, d_qk], dkv [s_kv, d_qk] (overwritten), dsink FP32 [H]
 *   (overwritten; required when sink is given, ignored otherwise).
 * Requires H a multiple of 64, d_qk 512 or 576, d_v 512, topk >= 1,
 * s_q, s_kv >= 1, s_q H d_qk and s_kv d_qk below 2^31, 16-byte aligned
 * tensors (4-byte for lse, sink, dsink, topk_idx, topk_len), and a workspace
 * of attn_dsa_bwd_workspace_size() bytes, 256-byte aligned (the FP32 dkv
 * accumulator).  Queues two kernels (after two memsets).  Returns a status
 * before any launch on bad arguments.
 */
ATTN_API size_t attn_dsa_bwd_workspace_size(int s_kv, int d_qk);
ATTN_API attn_status_t attn_dsa_bwd(const void *q, const void *kv, const void *o, const void *dout,
                                    const float *lse, const float *sink, const int *topk_idx,
                                    const int *topk_len, void *dq, void *dkv, float *dsink,
                                    void *workspace, size_t workspace_bytes, int s_q, int s_kv,
                                    int H, int d_qk, int d_v, int topk, float scale, int causal,
                                    void *stream);

/* Static string naming a status code. */
ATTN_API const char *attn_status_string(attn_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a kernel wait gave up;
 * its outputs are incomplete), ATTN_ERR_INVALID_ARG (packed-sequence offsets
 * that broke the rules of attn_fwd_layout; those sequences were skipped) or
 * ATTN_ERR_CUDA (the synchronisation failed, or a kernel could not align its
 * shared memory and wrote nothing).
 */
ATTN_API attn_status_t attn_last_device_error(void *stream);

/* Number of kernel launches the most recent attn_fwd* / attn_bwd* call on
 * this host thread queued (0 after a rejected call). */
ATTN_API int attn_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
