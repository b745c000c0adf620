/*
 * fa2.h -- C ABI of the GB300 (sm_103a) exact tiled attention: forward pass,
 * its backward pass and a decoding-regime forward.
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
 * Entry points:
 *   fa2_fwd / fa2_bwd        contiguous [B, H, N, d] tensors (fp16 or bf16),
 *                            lse [B, H, N] float32, full or causal attention;
 *   fa2_fwd_ex / fa2_bwd_ex  any strides, N_q != N_k, band and prefix masks,
 *                            packed variable-length batches (fa2_fwd_params);
 *   fa2_decode               up to FA2_DECODE_MAX_Q query rows per sequence
 *                            against long key sequences (fa2_fwd_params);
 *   fa2_fwd_host[_noalloc]   the forward on host buffers, end to end.
 *
 * Ownership: the caller owns every buffer.  fa2_fwd and fa2_fwd_ex allocate
 * no device memory; fa2_bwd, fa2_bwd_ex and fa2_decode take a caller
 * workspace.  The library keeps one small device status word per device for
 * reporting kernel-side wait timeouts and rejected packed offsets (see
 * fa2_get_device_status).
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
  FA2_ERR_SCRATCH_LIMIT = 6,  /* problem too large for fa2_fwd_host_noalloc's static scratch */
  FA2_ERR_DEVICE_SEQLENS = 7  /* packed-batch offsets out of range (fa2_get_device_status) */
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
 *   scale   : any finite value (0: uniform weights over the visible keys; a
 *             negative scale reverses the score order); the pages use 1/sqrt(d)
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
 * fa2_fwd_params -- arguments of fa2_fwd_ex, the general forward pass:
 * strided layouts, unequal query and key lengths, band and prefix masks and
 * packed variable-length batches.
 *
 * Which keys a query sees (the additive 0 / -inf mask of the Flash Attention
 * 2 page, "Causal masking", Option A, with the key tiles the mask removes
 * entirely skipped): in a sequence of N_q queries and N_k keys, query i is
 * aligned with key i + off, off = N_k - N_q (the last query with the last
 * key), and sees key j (0 <= j < N_k) iff
 *
 *     j < prefix_len,  or
 *     i + off - window_left <= j <= i + off + window_right
 *
 * where a window of -1 is unbounded on that side.  So (-1, -1) is full
 * attention, (-1, 0) causal (j <= i when N_q = N_k), (w, 0) a sliding window
 * of the w keys before each query and itself, and (-1, 0) with prefix_len = P
 * a prefix-LM (the first P keys visible to every query).  A query that sees
 * no key gets O = 0 and LSE = -inf.
 *
 * Element (b, h, i, c) of a tensor X in {q, o} is at
 *   X + b*X_strides[0] + h*X_strides[1] + (r0 + i)*X_strides[2] + c
 * elements, and of k, v likewise with key rows; lse (b, h, i) is at
 *   lse + b*lse_strides[0] + h*lse_strides[1] + (r0 + i).
 * Unpacked batches: r0 = 0, i < seqlen_q, j < seqlen_k.  Packed batches
 * (cu_seqlens_q and cu_seqlens_k both set): sequence b's query rows are
 * cu_seqlens_q[b] <= r < cu_seqlens_q[b+1] of q/o/lse (r0 = cu_seqlens_q[b])
 * and its keys cu_seqlens_k[b] <= r < cu_seqlens_k[b+1] of k/v; the batch
 * strides are ignored.
 */
typedef struct fa2_fwd_params {
  const void* q;          /* device, `dtype`, 16-byte aligned; read only */
  const void* k;          /* device, `dtype`, 16-byte aligned; read only */
  const void* v;          /* device, `dtype`, 16-byte aligned; read only */
  void* o;                /* device, `dtype`, 16-byte aligned; written */
  float* lse;             /* device, float32, 4-byte aligned; written (natural log) */
  int batch;              /* B >= 1 (packed: number of sequences) */
  int heads;              /* H >= 1 */
  int seqlen_q;           /* N_q >= 1 (packed: the longest sequence's query count) */
  int seqlen_k;           /* N_k >= 1 (packed: ignored) */
  int head_dim;           /* d: 64, 128 or 256 */
  int dtype;              /* FA2_FP16 or FA2_BF16 */
  float scale;            /* any finite value */
  int window_left;        /* >= 0, or -1 = unbounded */
  int window_right;       /* >= 0, or -1 = unbounded */
  int prefix_len;         /* >= 0 */
  int64_t q_strides[3];   /* batch, head, row strides in elements; multiples of 8 */
  int64_t k_strides[3];   /*   (a stride of a dimension of size 1 is ignored) */
  int64_t v_strides[3];
  int64_t o_strides[3];
  int64_t lse_strides[2]; /* batch, head strides in elements (row stride 1); >= 0 */
  const int* cu_seqlens_q; /* device, [batch + 1] int32 row offsets, or NULL */
  const int* cu_seqlens_k; /* device, [batch + 1] int32 row offsets, or NULL */
  int total_q;            /* packed: rows of q, o and lse (>= 1); else ignored */
  int total_k;            /* packed: rows of k and v (>= 1); else ignored */
} fa2_fwd_params;

/* sizeof(fa2_fwd_params) as compiled into the library (binding check). */
size_t fa2_fwd_params_size(void);

/*
 * fa2_fwd_ex -- the forward pass for fa2_fwd_params (asynchronous on
 * `stream`).  Same arithmetic and kernels as fa2_fwd, which is the special
 * case of contiguous [B,H,N,d] tensors, N_q = N_k = N, no prefix and
 * window (-1, causal ? 0 : -1).
 *
 * Checks before any launch: sizes, dtype, head dim, scale and windows as
 * documented above (FA2_ERR_INVALID_ARG / FA2_ERR_UNSUPPORTED); pointers
 * non-null and aligned and strides of dimensions larger than 1 positive
 * multiples of 8 elements below 2^39 (FA2_ERR_MISALIGNED for alignment,
 * FA2_ERR_INVALID_ARG otherwise); the byte ranges o and lse can touch
 * overlap neither each other nor those of q, k and v (FA2_ERR_INVALID_ARG);
 * only one of cu_seqlens_q / cu_seqlens_k set (FA2_ERR_INVALID_ARG).  The
 * caller keeps o's elements distinct (no two (b,h,i,c) at one address).
 *
 * Packed offsets live on the device and are checked by the kernel: a
 * sequence with cu_seqlens_q[b] > cu_seqlens_q[b+1], an offset outside
 * [0, total_q] (or [0, total_k] for keys), or more than seqlen_q queries is
 * left unwritten and the next fa2_get_device_status returns
 * FA2_ERR_DEVICE_SEQLENS.  The other sequences are written, except where
 * such offsets make in-range sequences' query rows overlap: a batch of at
 * most 192 sequences launches one CTA per real 128-row tile (as many as
 * non-overlapping sequences can hold), and tiles past that are skipped.
 * Rows of k and v outside a sequence may be read
 * (key tiles are 128 rows) and are multiplied by P = 0, so they must hold
 * finite values; rows past total_k read as zero.  Deterministic.
 */
int fa2_fwd_ex(const fa2_fwd_params* params, void* stream);

/* Query rows per sequence fa2_decode takes. */
#define FA2_DECODE_MAX_Q 8

/*
 * fa2_decode -- the forward pass for few query rows against many keys (the
 * decoding regime: a new token, or up to FA2_DECODE_MAX_Q of them, attending
 * to a long key/value cache).  Lesson 6.6 ("Common misconceptions") notes
 * that single-row decoding needs its own kernel: with one query row there is
 * no tile to fill a tensor core and the step is bound by reading K and V.
 * The keys of each (batch, head) are split into chunks reduced by separate
 * CTAs to online-softmax states (m, l, O~) that a second kernel merges with
 * the rescaling step of the tiled loop (Lesson 6.6, "Online softmax").
 * At d = 128 (and at d = 64 from two query rows on) the tiled tensor-core
 * kernel reduces each chunk for the whole query tile; one row at d = 64, and
 * d = 256, run the chunks on CUDA cores.
 *
 * Arguments as fa2_fwd_ex (same struct, masks, strides and packed batches),
 * with seqlen_q <= FA2_DECODE_MAX_Q (FA2_ERR_UNSUPPORTED otherwise; packed:
 * every sequence's query count) and seqlen_k the key count (packed: the
 * longest sequence's key count -- it sizes the split grid, which covers at
 * least that many keys; a sequence with more keys than the grid covers is
 * left unwritten and reported as FA2_ERR_DEVICE_SEQLENS).
 * `workspace`: device, >= fa2_decode_workspace_bytes(params) bytes, 256-byte
 * aligned, owned by the caller, overlapping no tensor; it holds fp32 partial
 * states and is written before it is read.  Asynchronous on `stream`; two
 * kernel launches (one when the keys fit a single chunk on the tensor-core
 * path).  Deterministic.
 */
int fa2_decode(const fa2_fwd_params* params, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace fa2_decode needs for these sizes (0 if they are invalid); it does
 * not depend on the device. */
size_t fa2_decode_workspace_bytes(const fa2_fwd_params* params);

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
 * current device's status word: FA2_OK, FA2_ERR_DEVICE_TIMEOUT if some
 * kernel's bounded wait on an mbarrier gave up (the kernel then abandoned its
 * tile, released its tensor memory and returned instead of hanging), else
 * FA2_ERR_DEVICE_SEQLENS if fa2_fwd_ex met out-of-range packed offsets.
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
 *   d                : 64, 128 or 256 (at d = 256 each 128-key tile runs as two
 *                      CTAs, one per half of the head dimension, that both
 *                      rebuild the tile's S and dP)
 *   other arguments  : as fa2_fwd
 *
 * dK and dV are each written once; dQ is accumulated over key tiles with
 * fp32 reduce-adds in L2 (TMA), so its last bits may vary between runs.
 * Outputs and workspace must not overlap any input or each other.  This is
 * fa2_bwd_ex for contiguous tensors and window (-1, causal ? 0 : -1).
 */
int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
            void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
            int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/* Device workspace fa2_bwd needs: fp32 [B,H,N,d] + fp32 [B,H,N], each 256-byte aligned. */
size_t fa2_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa2_bwd_params / fa2_bwd_ex -- gradients of fa2_fwd_ex: the same masks
 * (band, prefix), unequal query / key lengths, strided layouts and packed
 * batches.  `fwd` holds the forward call's arguments (q, k, v; o and lse
 * are the forward's outputs and are read here); the gradients share the
 * layouts of their primal tensors: dout and dq/dk/dv use o's, q's, k's and
 * v's strides.  head_dim 64, 128 or 256 (FA2_ERR_UNSUPPORTED otherwise).  Packed
 * batches: fwd.seqlen_k is the longest sequence's key count (it sizes the
 * grid; a sequence with more keys is left unwritten and reported as
 * FA2_ERR_DEVICE_SEQLENS; out-of-range offsets behave as in fa2_fwd_ex,
 * with key tiles in place of query tiles), and rows of dq outside every
 * sequence are set to
 * zero.  A key no query row sees gets dK = dV = 0; a query row that sees no
 * key gets dQ = 0.
 *
 * `workspace`: device, >= fa2_bwd_ex_workspace_bytes(&fwd) bytes, 256-byte
 * aligned: the fp32 dQ accumulator and D per row of every (batch, head)
 * slice, written before read.  dq, dk, dv and the workspace overlap no input
 * and no other output.  Asynchronous on `stream` (three kernels); dQ is
 * accumulated with fp32 reduce-adds, so its last bits may vary between runs.
 */
typedef struct fa2_bwd_params {
  fa2_fwd_params fwd;
  const void* dout;       /* device, o's layout, 16-byte aligned */
  void* dq;               /* device, q's layout, written */
  void* dk;               /* device, k's layout, written */
  void* dv;               /* device, v's layout, written */
  void* workspace;
  size_t workspace_bytes;
} fa2_bwd_params;

size_t fa2_bwd_ex_workspace_bytes(const fa2_fwd_params* fwd);
int fa2_bwd_ex(const fa2_bwd_params* params, void* stream);

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
