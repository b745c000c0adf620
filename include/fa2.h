/*
 * fa2.h -- C ABI of the GB300 (sm_103a) exact tiled attention forward pass.
 *
 * The operation (FlashAttention V2 in depth, section 6.1 "Full forward
 * algorithm"; Flash Attention 2 page, "Standard Attention" and "Causal
 * masking"): for every batch b and head h, with S = scale * Q K^T and, when
 * causal, S_ij = -inf for key j > query i,
 *
 *     O   = softmax_row(S) V                      (exact, not approximate)
 *     LSE = m + ln(l),  m = rowmax(S),  l = rowsum(exp(S - m))
 *
 * computed in query tiles that stream key/value tiles through on-chip memory
 * with an online softmax, so the N x N score matrix never reaches global
 * memory.  LSE is the natural-log logsumexp that section 7.1 keeps for the
 * backward pass.
 *
 * Layouts (all contiguous, row-major):
 *   q, k, v, o : [B, H, N, d] elements of `dtype` (fp16 or bf16)
 *   lse        : [B, H, N] float32
 *
 * Ownership: the caller owns every buffer.  fa2_fwd allocates no device
 * memory; the library keeps one small device status word per device for
 * reporting kernel-side wait timeouts (see fa2_get_device_status).
 *
 * No C++ exception crosses this interface: every entry point returns an
 * fa2_status code.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and o. */
typedef enum { FA2_FP16 = 0, FA2_BF16 = 1 } fa2_dtype;

typedef enum {
  FA2_OK = 0,
  FA2_ERR_INVALID_ARG = 1,    /* bad size, dtype, scale, null pointer or aliasing */
  FA2_ERR_UNSUPPORTED = 2,    /* head dim not in {64, 128, 256}, or no sm_103 device */
  FA2_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
  FA2_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  FA2_ERR_DEVICE_TIMEOUT = 5, /* a kernel wait ran out of time (fa2_get_device_status) */
  FA2_ERR_SCRATCH_LIMIT = 6   /* problem too large for fa2_fwd_host_noalloc's static scratch */
} fa2_status;

/*
 * fa2_fwd -- forward pass on device buffers (asynchronous on `stream`).
 *
 *   q, k, v : device pointers, [B, H, N, d] `dtype`, read only, 16-byte aligned
 *   o       : device pointer, [B, H, N, d] `dtype`, written (RN-even from fp32)
 *   lse     : device pointer, [B, H, N] float32, written (natural log)
 *   B, H, N : batch, heads, sequence length (each >= 1; B*H*N*d < 2^31 elements
 *             per tensor is not required, but B*H < 2^31 and N < 2^31 are)
 *   d       : head dimension, one of 64, 128, 256 (the pages cap head dim at 256)
 *   scale   : finite and > 0; the pages use 1/sqrt(d)
 *   causal  : 0 = every key visible; 1 = key j visible to query i iff j <= i
 *   dtype   : FA2_FP16 or FA2_BF16
 *   stream  : a cudaStream_t (0 = legacy default stream)
 *
 * Every argument is checked before any CUDA call; a bad argument returns its
 * code and launches nothing.  o and lse must not overlap q, k or v.  The call
 * does not synchronise; kernel-side failures surface through
 * fa2_get_device_status.  The result is deterministic (no atomics; every
 * output element is written once).
 */
int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
            int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * fa2_fwd_host -- the same forward pass on HOST buffers, end to end.
 *
 * Copies q, k, v (host, [B,H,N,d] `dtype`; pinned memory gives full copy
 * bandwidth) into the caller's device workspace, runs fa2_fwd on `stream`,
 * copies o and lse back into the host buffers and synchronises before
 * returning.  `workspace` is a device buffer of at least
 * fa2_fwd_host_workspace_bytes(B,H,N,d) bytes, 256-byte aligned, owned by the
 * caller.  Returns FA2_ERR_DEVICE_TIMEOUT if a kernel wait timed out.
 *
 * Problems with at least 48 MB of input are cut into up to 8 groups of
 * (b,h) slices: the copy-in of the next group and the copy-out of the
 * previous one run on two copy streams the library creates once per device
 * while the forward pass of the current group runs on `stream` (which first
 * waits for work already queued on it).  Such calls on one device are
 * serialised by the library.  Results are identical to the unsplit pass.
 */
int fa2_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                 float* lse_host, void* workspace, size_t workspace_bytes,
                 int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/* Device workspace fa2_fwd_host needs: q, k, v, o and lse, each 256-byte aligned. */
size_t fa2_fwd_host_workspace_bytes(int B, int H, int N, int d);

/* Bytes of the library's static device scratch used by fa2_fwd_host_noalloc. */
#define FA2_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fa2_fwd_host_noalloc -- fa2_fwd_host for callers that cannot allocate
 * device memory.  The pages have no counterpart: it exists for callers that
 * hold only host buffers and are not allowed to call cudaMalloc -- e.g. a
 * process whose device memory is wholly reserved by another allocator, so a
 * raw cudaMalloc would fail, or a latency-bound loop that must not call an
 * allocator that may synchronise the device.
 *
 * Same arguments and results as fa2_fwd_host, without the workspace: the
 * device staging copies of q, k, v, o and lse live in one static device
 * array of FA2_NOALLOC_SCRATCH_BYTES bytes that the library defines, which
 * every GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc or cudaFree, no allocating library call).
 *
 *   Limit: fa2_fwd_host_workspace_bytes(B, H, N, d) must not exceed
 *   FA2_NOALLOC_SCRATCH_BYTES; larger problems return FA2_ERR_SCRATCH_LIMIT
 *   before any CUDA call.
 *
 * The first call on a device looks up the array's device address on that
 * device (with it current); make that first call before any stream capture.
 * All calls on a device share the one array: calls whose work overlaps on
 * the GPU (other streams, other host threads) race and must be serialised by
 * the caller.  Nothing in the array needs to start at zero -- every byte a
 * call reads was written earlier in that same call.  The call synchronises
 * `stream` before returning.
 */
int fa2_fwd_host_noalloc(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                         float* lse_host, int B, int H, int N, int d, float scale, int causal, int dtype,
                         void* stream);

/*
 * fa2_get_device_status -- synchronises `stream`, then returns and clears the
 * current device's status word: FA2_OK, or FA2_ERR_DEVICE_TIMEOUT if some
 * kernel's bounded wait on an mbarrier gave up (the kernel then abandoned its
 * tile, released its tensor memory and returned instead of hanging).
 * `detail` (may be NULL) receives the raw status bits (role and wait site).
 */
int fa2_get_device_status(void* stream, uint32_t* detail);

/*
 * fa2_bwd -- gradients of fa2_fwd for an upstream gradient dout
 * (FlashAttention V2 in depth, section 7: P = exp(S - L) rebuilt from the
 * forward's logsumexp, dV = P^T dO, dP = dO V^T, D_i = rowsum(dO_i o O_i),
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q).  Asynchronous on
 * `stream`.
 *
 *   q, k, v, o, dout : device, [B,H,N,d] `dtype` (o is fa2_fwd's output)
 *   lse              : device, [B,H,N] float32, fa2_fwd's logsumexp
 *   dq, dk, dv       : device, [B,H,N,d] `dtype`, written
 *   workspace        : device, >= fa2_bwd_workspace_bytes(B,H,N,d) bytes,
 *                      256-byte aligned, owned by the caller: an fp32 dQ
 *                      accumulator [B,H,N,d] and D [B,H,N], both written
 *                      before they are read
 *   d                : 64 or 128 (FA2_ERR_UNSUPPORTED otherwise)
 *   other arguments  : as fa2_fwd
 *
 * dK and dV are each written once; dQ is accumulated over key tiles with
 * fp32 atomic adds, so its last bits may vary between runs.  Outputs and
 * workspace must not overlap any input or each other.
 */
int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
            void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
            int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/* Device workspace fa2_bwd needs: fp32 [B,H,N,d] + fp32 [B,H,N], each 256-byte aligned. */
size_t fa2_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa2_selftest_wait_timeout -- exercises the kernels' failure path without a
 * GPU fault: launches one CTA whose single wait, made through the same
 * bounded-wait routine every forward-kernel wait uses, is on an mbarrier that
 * nothing ever completes.  After `limit_us` microseconds (1 .. 1e6) the wait
 * gives up, records its site in the device status word and the kernel
 * returns normally.  Asynchronous on `stream`; a following
 * fa2_get_device_status returns FA2_ERR_DEVICE_TIMEOUT (detail bit 8 + 11)
 * and clears the word.  No counterpart on the pages: it tests the library's
 * own hang protection (FlashAttention V2 in depth describes no failure
 * handling).
 */
int fa2_selftest_wait_timeout(int limit_us, void* stream);

/* Static English description of a status code. */
const char* fa2_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int fa2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */
