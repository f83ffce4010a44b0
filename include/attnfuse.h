/*
 * libattnfuse — causal softmax attention with Rotary Position Embedding (RoPE), forward and
 * backward, for NVIDIA GB300 (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * The operation.  "AttnFuse Makes RoPE a First-Class Attention Compilation Operation" (2026-09-13
 * AI papers report), paragraphs 1-2, and the AttnFuse abstract (arxivdaily 2609.13612): RoPE is a
 * transformation of Q and K applied before the QK^T product, composed with the causality and
 * softmax building blocks into one fused kernel.  Paragraphs 3-5 of the same report weigh that
 * fused form against rotating Q and K in a separate pass first ("pre-rotation"), whose cost is
 * memory bandwidth where the fused form's is compute; both forms are offered here, and a third that
 * the GB300 measurements favour for grouped-query attention (K rotated in a pass, Q on chip: see
 * ATTNFUSE_SPLIT).  The pages print no formula; this library fixes:
 *     theta_k = rope_base^(-2k/d), k = 0 .. d/2-1, pairs (k, k + d/2), position = token index,
 *     x'[k] = x[k] cos(p theta_k) - x[k+d/2] sin(p theta_k),
 *     x'[k+d/2] = x[k+d/2] cos(p theta_k) + x[k] sin(p theta_k)       (Q and K; V is not rotated)
 *     out[b,i,h,:] = sum_{j<=i} softmax_j(q'_{b,i,h} . k'_{b,j,h/g} / sqrt(d)) v[b,j,h/g,:]
 *     lse[b,h,i]   = ln sum_{j<=i} exp(q'.k'/sqrt(d))                   (natural log)
 * with g = Hq / Hkv (grouped-query attention: consecutive query heads share a KV head).
 *
 * Layout (row-major, contiguous, element type per `dtype`):
 *     q, out : [B, N, Hq, d]        k, v : [B, N, Hkv, d]        lse : [B, Hq, N] float32
 * Supported: d in {64, 128}; bf16 or fp16; B, N, Hq, Hkv >= 1; Hq % Hkv == 0; N < 2^24.
 * Arithmetic: rotation and softmax statistics in fp32, products on the tensor cores with fp32
 * accumulation; P and the rotated Q/K are rounded to `dtype` once.
 *
 * Ownership and streams.  Every buffer belongs to the caller and must be device memory (q, k, v,
 * out, workspace 16-byte aligned; lse 4-byte aligned).  `stream` is a cudaStream_t passed as void*
 * (so that this header needs no CUDA include; NULL = the legacy default stream); all work is
 * enqueued on it and the calls return without waiting.  `rope_base` is a double because theta_k is
 * computed from it in fp64.
 *
 * Errors.  Arguments are validated before anything is launched; a failed call returns a status,
 * launches nothing and leaves a message for attnfuse_last_error().  Faults raised while kernels
 * run surface at the caller's next synchronisation.  Every barrier wait inside the kernels is
 * bounded: if one runs out, the kernel stops, records it in a device status word that
 * attnfuse_device_status() reads, and returns (later launches then do nothing until it is read).
 */
#ifndef ATTNFUSE_H_
#define ATTNFUSE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTNFUSE_FUSED = 0,
  ATTNFUSE_PREROTATE = 1,
  ATTNFUSE_AUTO = 2,
  ATTNFUSE_SPLIT = 3,
  ATTNFUSE_NONE = 4
} attnfuse_mode_t;

typedef enum { ATTNFUSE_BF16 = 0, ATTNFUSE_FP16 = 1 } attnfuse_dtype_t;

typedef enum {
  ATTNFUSE_OK = 0,
  ATTNFUSE_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, workspace too small */
  ATTNFUSE_ERR_UNSUPPORTED = 2, /* d not in {64,128}, device is not compute capability 10.3 */
  ATTNFUSE_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the CUDA error) */
  ATTNFUSE_ERR_TIMEOUT = 4,     /* a kernel barrier wait ran out (attnfuse_device_status) */
  ATTNFUSE_ERR_NO_MEMORY = 5    /* workspace allocation failed */
} attnfuse_status_t;

/*
 * Causal RoPE attention forward.
 *   mode = ATTNFUSE_FUSED:     one kernel; Q and K tiles are rotated in shared memory.
 *   mode = ATTNFUSE_PREROTATE: a RoPE pass writes rotated Q', K' into `workspace`, then the same
 *                              attention kernel runs on Q', K', V without rotation.
 *   mode = ATTNFUSE_SPLIT:     a RoPE pass writes rotated K' into `workspace` (K is re-read by every
 *                              query tile that needs it), then the attention kernel rotates each
 *                              query tile on chip (each is read once): rotation cost paid once per
 *                              element for both tensors.
 *   mode = ATTNFUSE_AUTO:      whichever mode attnfuse_select_mode returns for the shape.
 *   mode = ATTNFUSE_NONE:      no rotation: q and k are taken as already rotated (e.g. by
 *                              attnfuse_rope_apply) and the attention kernel of the pre-rotate path
 *                              runs on them alone -- the "plain causal attention" that follows the
 *                              standalone RoPE pass in the pages' pre-rotation path.  Takes kv_len
 *                              but no rotation option (rotary_dim, interleaved, positions).
 * FUSED and AUTO calls with few queries per KV head -- (Hq / Hkv) N <= 16 query rows (a decode
 * step, a speculative-decode step) -- run split-KV decode kernels instead: each CTA rotates one
 * slice of one KV head's keys and the head's query rows on chip and runs the two products as
 * 16-row tensor-core tiles; a second kernel merges the slices' partial softmax sums.
 * All modes compute the function in the header comment.  `lse` may be NULL (not written).
 * `workspace` must hold attnfuse_workspace_bytes(...) bytes (0 for FUSED outside the decode
 * shapes); if it is NULL while
 * bytes are needed, the call allocates with cudaMallocAsync and frees with cudaFreeAsync on
 * `stream`.  Query rows never read keys beyond their own position; rows are independent.
 */
attnfuse_status_t attnfuse_rope_causal_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                           int Hq, int Hkv, int N, int d, double rope_base, attnfuse_mode_t mode,
                                           attnfuse_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                           void* stream);

/* Bytes of workspace attnfuse_rope_causal_fwd needs: 0 for FUSED and NONE; for PREROTATE the rotated copies
 * of Q and K (each rounded up to 256 bytes); for SPLIT the rotated K; for AUTO those of the selected
 * mode; for FUSED and AUTO at the decode shapes the decode kernels' partial results (per key
 * slice and KV head, 16 query-row slots of d + 2 floats).  Returns 0 for invalid arguments. */
size_t attnfuse_workspace_bytes(int B, int Hq, int Hkv, int N, int d, attnfuse_mode_t mode, attnfuse_dtype_t dtype);

/*
 * The fastest mode for a shape on GB300, from the measured sweep of all three ("Rotation Calculus" in
 * "AttnFuse Makes RoPE a First-Class Attention Compilation Operation", paragraph 2, made a runtime
 * choice): grouped-query attention (Hq / Hkv >= 2) with N >= 1024 -> SPLIT (fastest at all 14
 * measured points from 1024 to 16384); multi-head attention (Hq == Hkv) with N >= 4096 -> SPLIT
 * (tied with pre-rotation at 4096, ahead from 5500), with 1892 <= N < 4096 -> PREROTATE (measured
 * N* = 1892 against FUSED); else -> FUSED.
 * Host-only and pure: no device access; arguments it cannot classify (non-positive sizes, Hq not a
 * multiple of Hkv) give FUSED.
 */
attnfuse_mode_t attnfuse_select_mode(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype);

/*
 * RoPE alone (the pre-rotation pass): y = RoPE(x) for x, y of shape [B, N, H, d], position of
 * (b, n) = n.  y may equal x (in place); otherwise the two must not overlap.  Bounded by HBM
 * bandwidth: it reads and writes every element once.
 */
attnfuse_status_t attnfuse_rope_apply(const void* x, void* y, int B, int N, int H, int d, double rope_base,
                                      attnfuse_dtype_t dtype, void* stream);

/*
 * RoPE variants and the general causal form (extensions of the rotation and the causality block the
 * pages name, "AttnFuse Makes RoPE a First-Class Attention Compilation Operation", paragraphs 1-2;
 * the pages fix no pairing, rotary dimension, key length or position source).
 *   rotary_dim: only entries [0, r) of each head vector are rotated, with theta_k = base^(-2k/r),
 *               k < r/2; entries [r, d) pass through unchanged.  0 means r = d.  Otherwise
 *               16 <= r <= d and r a multiple of 16.
 *   interleaved: 0 pairs (k, k + r/2) (half-split, the default form); 1 pairs (2k, 2k + 1).
 *   kv_len:     Nk, the number of key/value tokens per batch entry (k, v are [B, Nk, Hkv, d]); 0
 *               means N.  Otherwise N <= Nk < 2^24.  The N queries are the last N of the Nk tokens
 *               (a prefill that extends a cache of Nk - N earlier tokens; N = 1 is one decode
 *               step): query i sees keys j <= Nk - N + i.
 *   q_positions: NULL, or device int32 [B, N] (4-byte aligned): the rotation position of each
 *               query token.  NULL means Nk - N + i.
 *   k_positions: NULL, or device int32 [B, Nk]: the rotation position of each key token.  NULL
 *               means j.  Positions may be any int32 values; they set the RoPE angles only, never
 *               the mask.  The fused kernel computes exact cos/sin per row when positions are given
 *               (slower than the default walk along consecutive positions).
 * A NULL pointer to the struct means all zero: the functions without _ex.
 */
typedef struct {
  int rotary_dim;
  int interleaved;
  int kv_len;
  const int32_t* q_positions;
  const int32_t* k_positions;
} attnfuse_rope_opts_t;

/* attnfuse_workspace_bytes for attnfuse_rope_causal_fwd_ex with `opts` (may be NULL): the rotated K
 * has kv_len tokens.  Returns 0 for invalid arguments. */
size_t attnfuse_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, attnfuse_mode_t mode, attnfuse_dtype_t dtype,
                                   const attnfuse_rope_opts_t* opts);

/* attnfuse_rope_causal_fwd with a RoPE variant and/or the general causal form (opts may be NULL);
 * same arguments otherwise (N = query tokens; `lse` is [B, Hq, N]).  Invalid opts give
 * ATTNFUSE_ERR_INVALID_ARG.  In PREROTATE mode the workspace must hold
 * attnfuse_workspace_bytes_ex(...) bytes (rotated Q [B, N, Hq, d] and K [B, Nk, Hkv, d]); AUTO
 * applies attnfuse_select_mode with Nk in place of N. */
attnfuse_status_t attnfuse_rope_causal_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                                              int B, int Hq, int Hkv, int N, int d, double rope_base,
                                              attnfuse_mode_t mode, attnfuse_dtype_t dtype, void* workspace,
                                              size_t workspace_bytes, const attnfuse_rope_opts_t* opts,
                                              void* stream);

/* attnfuse_rope_apply with a RoPE variant (opts may be NULL).  Out of place, the entries that are
 * not rotated are copied to y; in place they are left as they are.  opts->q_positions, if not NULL,
 * gives the position of each token of x ([B, N] int32); kv_len must be 0 and k_positions NULL. */
attnfuse_status_t attnfuse_rope_apply_ex(const void* x, void* y, int B, int N, int H, int d, double rope_base,
                                         attnfuse_dtype_t dtype, const attnfuse_rope_opts_t* opts, void* stream);

/*
 * Backward pass of attnfuse_rope_causal_fwd (N queries and keys, positions i and j, half-split
 * rotation over all d entries): the gradients of a loss L with respect to q, k and v, given
 * dout = dL/dout and the forward's out and lse ("AttnFuse Makes RoPE a First-Class Attention
 * Compilation Operation", paragraph 3, names the training step this serves; the chain rule through
 * paragraphs 1-2's rotation, causal mask and softmax).  With q' = R(i) q, k' = R(j) k,
 * P = softmax(q'k'^T / sqrt(d)) causal and D_i = dout_i . out_i:
 *     dv = P^T dout,  dS = P o (dout v^T - D),  dq = R^T (dS k' / sqrt(d)),  dk = R^T (dS^T q' / sqrt(d))
 * (GQA: a KV head's dk, dv sum over its query heads; L's dependence on lse is not propagated).
 * Layouts as the forward: q, out, dout, dq [B, N, Hq, d]; k, v, dk, dv [B, N, Hkv, d]; lse
 * [B, Hq, N] float32 (required).  Outputs must not overlap the inputs.  `workspace` holds
 * attnfuse_bwd_workspace_bytes(...) bytes (rotated q and k, D, a work counter) and serves one call
 * at a time; NULL allocates with cudaMallocAsync / cudaFreeAsync on `stream`.  Errors as for the
 * forward.
 */
attnfuse_status_t attnfuse_rope_causal_bwd(const void* q, const void* k, const void* v, const void* out,
                                           const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                           int Hq, int Hkv, int N, int d, double rope_base, attnfuse_dtype_t dtype,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* attnfuse_rope_causal_bwd for every option of attnfuse_rope_opts_t: the RoPE variants (rotary_dim,
 * interleaved), explicit positions (q_positions [B, N], k_positions [B, Nk]) and more keys than
 * queries (kv_len = Nk >= N: k, v, dk, dv are [B, Nk, Hkv, d], the N queries are the last N of the
 * Nk tokens and query i sees keys j <= Nk - N + i, as in the forward -- the backward of a prefill
 * that extends a cache).  For the half-split form over all d entries at the default positions the
 * kernels rotate the gradients back themselves; otherwise they produce them in the rotated frame
 * and a pre-rotation pass with the negated positions rotates dq and dk back (R^T).  `workspace`
 * holds attnfuse_bwd_workspace_bytes_ex(...) bytes. */
attnfuse_status_t attnfuse_rope_causal_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                                              const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                              int Hq, int Hkv, int N, int d, double rope_base, attnfuse_dtype_t dtype,
                                              void* workspace, size_t workspace_bytes,
                                              const attnfuse_rope_opts_t* opts, void* stream);

/* Bytes of workspace attnfuse_rope_causal_bwd needs (0 for invalid arguments). */
size_t attnfuse_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype);

/* Bytes of workspace attnfuse_rope_causal_bwd_ex needs with these options: rotated q [B, N, Hq, d],
 * rotated k [B, Nk, Hkv, d] (Nk = kv_len, 0 meaning N) and D [B, Hq, N] float, each rounded up to
 * 256 bytes, then 256 bytes for the dQ kernel's work counter (0 for invalid arguments).  One
 * workspace serves one call at a time: calls in flight together on different streams need their
 * own. */
size_t attnfuse_bwd_workspace_bytes_ex(int B, int Hq, int Hkv, int N, int d, attnfuse_dtype_t dtype,
                                       const attnfuse_rope_opts_t* opts);

/*
 * Synchronises `stream`, then reads and clears the device status word.  Returns
 * ATTNFUSE_ERR_TIMEOUT if a kernel's barrier wait ran out since the last read, ATTNFUSE_ERR_CUDA if
 * synchronising failed (e.g. a device fault), ATTNFUSE_OK otherwise.
 */
attnfuse_status_t attnfuse_device_status(void* stream);

/*
 * Diagnostic for the timeout path: launches one CTA that waits on a barrier nothing arrives on and
 * gives up after `timeout_ns` nanoseconds (at most 1e9), setting the device status word as a real
 * timeout would.  Nothing faults; the context stays usable.
 */
attnfuse_status_t attnfuse_diag_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Size of the fixed scratch buffer behind attnfuse_rope_causal_fwd_prerotate_noalloc (64 MiB: the
 * rotated Q and K of the Llama-3-8B attention shape, B=1, N=4096, 32+8 heads, d=128, take 42 MB).
 */
#define ATTNFUSE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Pre-rotate forward that allocates nothing.  The AttnFuse pages have no counterpart to this call:
 * it exists for callers that cannot allocate device memory -- e.g. a framework whose own caching
 * allocator has reserved the GPU's memory, or code that must not risk an allocation failure or
 * stall in the middle of a step -- and that also cannot lend a workspace.
 *
 * Same arguments and result as attnfuse_rope_causal_fwd with mode = ATTNFUSE_PREROTATE, except that
 * the rotated Q and K go to a fixed buffer of ATTNFUSE_NOALLOC_SCRATCH_BYTES compiled into the
 * library (a __device__ array: every GPU that loads the library holds it until the process exits).
 * Calls whose rotated Q and K need more than that (attnfuse_workspace_bytes(..., PREROTATE, ...))
 * return ATTNFUSE_ERR_INVALID_ARG before launching anything; every other argument is checked as in
 * attnfuse_rope_causal_fwd, also before any device work.  No cudaMalloc, cudaFree or other
 * allocating call is made.  The first call on each device looks up the buffer's device address
 * (cudaGetSymbolAddress, with that device current), and so does the first call after the device's
 * context was destroyed and created again (e.g. cudaDeviceReset): make such a first call before any
 * stream capture.
 * All calls share the one buffer and it keeps the last call's contents: calls that may overlap on
 * the GPU (other streams, other host threads) race on it and must be ordered by the caller.
 */
attnfuse_status_t attnfuse_rope_causal_fwd_prerotate_noalloc(const void* q, const void* k, const void* v, void* out,
                                                              float* lse, int B, int Hq, int Hkv, int N, int d,
                                                              double rope_base, attnfuse_dtype_t dtype, void* stream);

/* Static description of a status code. */
const char* attnfuse_status_string(attnfuse_status_t status);

/* Detail of the last failure on the calling thread ("" if none). */
const char* attnfuse_last_error(void);

/* Library version string. */
const char* attnfuse_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNFUSE_H_ */
