/*
 * fa_fwd.h — C ABI of the exact attention forward pass for sm_103a (GB300).
 *
 * The operation (cited by page title and section):
 *   "Before implementing FlashAttention in Triton: FA1, 2 forward pass",
 *   "Why it is needed": S = Q K^T, P = softmax(S), O = P V, softmax along
 *   each row of S; the FA2 section: O_i = diag(l_i)^-1 O~_i and
 *   L_i = m_i + log l_i, with exp(S_ij - L_i) = P_ij.
 *   "How FlashAttention got past the O(N^2) memory wall", tiling loop:
 *   S_ij = Q_i K_j^T / sqrt(D); "v2 and v3": key blocks right of the query
 *   block are skipped under the causal mask.
 *   "FlashAttention: it was data movement, not compute, that made attention
 *   fast", "Must the N x N matrix be stored?": O = softmax(Q K^T / sqrt(d)) V.
 *
 * For every batch b, head h and query row i (all indices zero-based):
 *   s_ik = scale * sum_t Q[b,h,i,t] K[b,h,k,t]     for visible keys k
 *   L[b,h,i] = ln sum_k exp(s_ik)                   (natural log)
 *   O[b,h,i,:] = sum_k exp(s_ik - L[b,h,i]) V[b,h,k,:]
 * where every key is visible, or, when `causal` is nonzero, key k is visible
 * to query i iff k <= i.  No N x N matrix is ever written to memory.
 *
 * Conventions shared by every entry point:
 *   - Return value: FA_OK (0) or a negative fa_status.  An argument error is
 *     reported before anything is enqueued.
 *   - Device pointers refer to memory of the current CUDA device; the caller
 *     owns every buffer.  The library allocates no device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) and return once enqueued.
 *   - A device-side bounded wait that expires (a protocol fault, never
 *     expected) is recorded on the device and reported by fa_check_errors.
 */
#ifndef FA_FWD_H
#define FA_FWD_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad flag, aliasing */
  FA_ERR_UNSUPPORTED = -2, /* head dim other than 64/128, negative scale, too large */
  FA_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned (lse: 4-byte) */
  FA_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed; see fa_get_last_cuda_error */
  FA_ERR_TIMEOUT = -5      /* a bounded device-side wait expired (see fa_check_errors) */
} fa_status;

/*
 * fa_fwd — attention forward on device buffers.
 *
 *   q, k, v : bf16 [B, H, N, d], contiguous (d fastest), device, read only.
 *   o       : bf16 [B, H, N, d], contiguous, device, written (round to
 *             nearest even from fp32).
 *   lse     : fp32 [B, H, N], contiguous, device, written: L = ln sum exp(s)
 *             in the units of the scaled scores.
 *   B, H, N : >= 1.  Any N is accepted; a partial last tile is masked.
 *             B*H <= 2^31-1 and B*H*N*d < 2^62.
 *   d       : 64 or 128 (else FA_ERR_UNSUPPORTED).
 *   scale   : finite and >= 0 (negative: FA_ERR_UNSUPPORTED; non-finite:
 *             FA_ERR_INVALID_ARG).  Usually 1/sqrt(d).
 *   causal  : 0 (every key visible) or 1 (key index <= query index).
 *   stream  : cudaStream_t as void*.
 *
 * q, k, v, o must be 16-byte aligned and lse 4-byte aligned
 * (FA_ERR_MISALIGNED).  o and lse must not overlap q, k or v
 * (FA_ERR_INVALID_ARG).  Not reentrant on overlapping outputs; concurrent
 * calls on distinct buffers are safe.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_host — the same operation on HOST buffers, for callers whose data
 * lives in host memory.  Enqueues on `stream`: host-to-device copies of
 * q, k, v into the caller's device staging buffers dq, dk, dv; fa_fwd on
 * them into do_, dlse; device-to-host copies into o and lse.  Returns after
 * enqueueing; the host buffers must stay valid (and, for the copies to be
 * asynchronous, pinned) until the stream reaches that point.  Argument rules
 * as for fa_fwd, applied to the device buffers; host pointers must be
 * non-null.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* dq,
                void* dk, void* dv, void* do_, float* dlse, int B, int H, int N, int d,
                float scale, int causal, void* stream);

/*
 * fa_check_errors — synchronise `stream`, then report and clear the device
 * error record: FA_ERR_TIMEOUT if a bounded wait expired in any kernel since
 * the last check (the outputs of that call are then invalid), FA_ERR_CUDA if
 * the synchronisation failed, else FA_OK.
 */
int fa_check_errors(void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(int status);

/* The raw cudaError_t behind the most recent FA_ERR_CUDA on this thread. */
int fa_get_last_cuda_error(void);

/*
 * The device error record behind the most recent FA_ERR_TIMEOUT returned by
 * fa_check_errors on this thread: out4[0] = code (1 = bounded wait expired),
 * out4[1] = wait site, out4[2] = CTA index, out4[3] = work item.  All zero if
 * none.  FA_ERR_INVALID_ARG if out4 is NULL.
 */
int fa_get_last_error_record(unsigned int* out4);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_FWD_H */
