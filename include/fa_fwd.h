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

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad flag, aliasing */
  FA_ERR_UNSUPPORTED = -2, /* head dim other than 64/128, sizes too large; negative scale
                              in fa_bwd and fa_fwd_e4m3 */
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
 *   scale   : any finite value (non-finite: FA_ERR_INVALID_ARG); usually
 *             1/sqrt(d).  A negative scale is computed as S' = (-Q) K^T,
 *             the MMA negating its Q operand, with the positive constant
 *             |scale|, which gives the same scores scale * Q K^T exactly.
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
 * lives in host memory.  The heads are split into up to eight groups (with
 * four or more, the first and the last hold half the heads of the others,
 * since nothing overlaps the first upload or the last download),
 * pipelined over three streams of the library's own (created once per
 * device): uploads of each group's q, k, v rows into the caller's device
 * staging buffers dq, dk, dv, in group order; the forward of each group into
 * do_, dlse as soon as its inputs have landed; downloads of its O and L rows
 * into o and lse as soon as its kernel is done.  The pipeline is forked from
 * `stream` and joined back to it, so everything is ordered after earlier
 * work on `stream` and later work on `stream` sees the results.  Returns
 * after enqueueing; the host buffers must stay valid (and, for the copies to
 * be asynchronous, pinned) until `stream` reaches
 * that point.  Calls from several threads are serialised while they
 * enqueue.  Argument rules as for fa_fwd, applied to the device buffers;
 * host pointers must be non-null.  If an error occurs after work has been
 * queued on the internal streams, the call first waits for that work to
 * finish, then returns the error.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* dq,
                void* dk, void* dv, void* do_, float* dlse, int B, int H, int N, int d,
                float scale, int causal, void* stream);

/*
 * fa_fwd_splitkv — the same operation as fa_fwd, with the key blocks of each
 * 256-row query tile cut into up to num_splits ranges that run as separate
 * work units, for shapes whose query tiles alone cannot occupy the GPU
 * (small B*H with long N).  Each range leaves a normalised partial output
 * O_s (fp32) and its logsumexp L_s in `workspace`; a second kernel merges
 * them per row by the block-merge rule of the online softmax:
 *   L = m + ln sum_s exp(L_s - m),  m = max_s L_s,
 *   O = sum_s exp(L_s - L) O_s
 * ("FlashAttention: it was data movement, not compute, that made attention
 * fast", section "Softmax can be computed in pieces": partial sums taken
 * against a local maximum are rescaled by exp(m_local - m) before they are
 * added; the result equals the whole-row softmax).
 *
 *   q, k, v, o, lse, B, H, N, d, scale, causal, stream: as for fa_fwd.
 *   num_splits : 1..64 ranges per query tile; 0 picks
 *                fa_fwd_splitkv_num_splits.  A count above the key blocks of
 *                a tile, ceil(N / 256), is lowered to that number first (the
 *                units would be the same), and the workspace layout below
 *                uses the lowered count.  1 runs fa_fwd and needs no
 *                workspace.
 *   workspace  : device memory owned by the caller, 16-byte aligned, at
 *                least fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
 *                bytes, not overlapping q, k, v, o or lse.  Layout: fp32
 *                O_s [num_splits][B*H][N][d], then fp32 L_s [num_splits][B*H][N].
 *                Contents on entry are ignored; the call overwrites it.
 *   workspace_bytes : its size in bytes.
 *
 * Errors: as for fa_fwd; num_splits outside 0..64, a missing or too small
 * workspace, or overlap: FA_ERR_INVALID_ARG; an unaligned workspace:
 * FA_ERR_MISALIGNED.  Enqueues two kernels on `stream`.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, float scale, int causal, int num_splits, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Workspace bytes that suffice for fa_fwd_splitkv with these sizes and
 * num_splits >= 1: num_splits * B*H*N * (d + 1) * 4 (the call itself needs
 * this for min(num_splits, ceil(N / 256)) splits).  0 if an argument is out
 * of range.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);

/*
 * The split count num_splits = 0 selects on the current device: 1 when the
 * one-pass query tiles alone give every SM pair work; otherwise, among 1..8
 * (at most the key blocks of a tile), the count that minimises (waves of work
 * units over the SM pairs) x (key blocks of the longest unit + about 3 blocks
 * of fixed cost per unit), the smaller on ties.  FA_ERR_INVALID_ARG for
 * non-positive sizes.
 */
int fa_fwd_splitkv_num_splits(int B, int H, int N, int causal);

/*
 * fa_fwd_splitkv_noalloc — fa_fwd_splitkv without a caller workspace: the
 * partial results go to a fixed scratch array that is part of the library's
 * device image (fa_fwd_splitkv_noalloc_capacity() bytes per device), so the
 * call allocates nothing and needs no buffer beyond q, k, v, o and lse.
 * The pages have no counterpart to this entry point; it is a deployment
 * convenience around the same split forward.
 *
 *   Arguments: as for fa_fwd_splitkv, without workspace / workspace_bytes
 *   (num_splits is lowered to ceil(N / 256) the same way, before the
 *   capacity check).
 *   Errors: as for fa_fwd_splitkv; FA_ERR_UNSUPPORTED when the partials of
 *   this call (fa_fwd_splitkv_workspace_size of the lowered count) exceed
 *   the scratch capacity.
 *   Memory: the 64 MiB scratch is reserved on every device where the library
 *   is loaded, whether or not this entry point is ever called.
 *   Set-up: the first call on a device looks up that device's address of
 *   the scratch (cudaGetSymbolAddress, with the device current) and keeps
 *   it; make that first call before any stream capture on the device.
 *   The scratch is shared by every call on a device and keeps the last
 *   call's contents (each call overwrites what it reads): calls that may run
 *   at the same time (on different streams) race on it and must not both use
 *   this entry point; calls ordered on one stream are safe.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal, int num_splits,
                           void* stream);

/* Bytes of the fixed scratch fa_fwd_splitkv_noalloc may use per device. */
size_t fa_fwd_splitkv_noalloc_capacity(void);

/*
 * fa_bwd — attention backward: the gradients of L_total with respect to q,
 * k, v given dO = dL_total/dO, recomputing P blockwise from S and the
 * forward's logsumexp instead of storing it ("Before implementing
 * FlashAttention in Triton: FA1, 2 forward pass", FA2 section: L alone gives
 * the normalised P back; "How FlashAttention got past the O(N^2) memory
 * wall", "v2 and v3"; "FlashAttention: it was data movement, not compute,
 * that made attention fast", "The paradox that recomputing is cheaper").
 * With P_ik = exp(s_ik - L_i) on visible keys:
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_t dO_it O_it,  dS = P (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   q, k, v   : the forward's inputs, bf16 [B, H, N, d], device, read only.
 *   o, lse    : the forward's outputs (fa_fwd), read only.
 *   dout      : bf16 [B, H, N, d], device, the gradient of O, read only.
 *   dq, dk, dv: bf16 [B, H, N, d], device, written.
 *   B, H, N, d, scale, causal, stream: as for fa_fwd (the same values the
 *               forward ran with), except that scale must be >= 0 (negative:
 *               FA_ERR_UNSUPPORTED).
 *   workspace : device memory owned by the caller, 16-byte aligned, at least
 *               fa_bwd_workspace_size(B, H, N, d) bytes: the rows' -L log2 e
 *               and -D as two fp32 planes [B*H][Tp], Tp = N rounded up to a
 *               multiple of 128, then 256 bytes of work counters.  Contents
 *               on entry are ignored.
 *
 * Errors: as for fa_fwd; a null or unaligned (16 bytes) dout, dq, dk, dv or
 * workspace, a workspace that is too small, or any output (dq, dk, dv,
 * workspace) overlapping an input or another output: FA_ERR_INVALID_ARG or
 * FA_ERR_MISALIGNED.  Enqueues three kernels: D on `stream`, then dK and dV
 * (a key-outer walk) on `stream`, launched as a programmatic dependent of the
 * first (its set-up overlaps that kernel's end; it reads nothing the first
 * kernel writes before that kernel has completed), and dQ (a query-outer
 * walk that recomputes S and dP) on a stream of the library's own, forked
 * from `stream` after the first kernel and joined back to it (event record /
 * wait), so that the two walks share the GPU; work enqueued on `stream`
 * afterwards waits for all three.  Each gradient is accumulated on chip and
 * written once.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_bwd needs: B*H*Tp * 8 + 256 (Tp = N rounded up to a
 * multiple of 128); 0 for invalid sizes. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * 8-bit (E4M3) forward.  "How FlashAttention got past the O(N^2) memory
 * wall", section "v2 and v3", credits FP8 support with about twice the BF16
 * throughput and fixes nothing else; the format and scaling below are this
 * library's reading.  E4M3 is the OCP 8-bit floating point format (bias 7,
 * largest finite 448, no infinities).  Each (batch, head) slice of Q, K and
 * V has its own fp32 descale: the value a code stands for is
 * E4M3(code) * descale.  O and L are those of the exact attention of the
 * dequantised inputs up to the rounding of the softmax weights P~ to E4M3
 * inside the P~ V product (L does not see that rounding).
 *
 * fa_quantize_e4m3 — codes and descales of a bf16 tensor:
 *   x        : device, bf16 [B, H, N, d] contiguous, 16-byte aligned, finite.
 *   x8       : device, fa_e4m3_bytes(B, H, N, d, keys_last) bytes, 16-byte
 *              aligned.  keys_last = 0: codes [B, H, N, d]; keys_last = 1:
 *              codes [B, H, d, P] with P = N rounded up to a multiple of 16
 *              and columns N..P-1 set to 0 (the layout fa_fwd_e4m3 takes
 *              for V).
 *   descale  : device, fp32 [B, H], 4-byte aligned: amax / 448 per slice,
 *              amax = max |x| over the slice.  Codes are E4M3(x * s) with
 *              s = 448 / amax (s = 1 when amax = 0), rounded to nearest
 *              even, saturated at +-448, every step correctly rounded fp32.
 *   d        : 64 or 128; B * H <= 65535.
 * Errors: NULL pointer, B/H/N <= 0 or keys_last not 0/1: FA_ERR_INVALID_ARG;
 * other d or B * H: FA_ERR_UNSUPPORTED; unaligned: FA_ERR_MISALIGNED; x8 or
 * descale overlapping an input or each other: FA_ERR_INVALID_ARG.  Enqueues
 * a memset and three kernels on `stream`.
 */
size_t fa_e4m3_bytes(int B, int H, int N, int d, int keys_last);
int fa_quantize_e4m3(const void* x, void* x8, float* descale, int B, int H, int N, int d,
                     int keys_last, void* stream);

/*
 * fa_quantize_qkv_e4m3 — fa_quantize_e4m3 of q and k (keys_last = 0) and of
 * v (keys_last = 1) in one call: the same codes and descales, in four
 * launches instead of twelve.  q8, k8 and vt8 are sized as fa_e4m3_bytes
 * gives; the descale arrays are fp32 [B, H] each.  Errors as for
 * fa_quantize_e4m3; besides, no output may overlap another output or an
 * input (FA_ERR_INVALID_ARG).
 */
int fa_quantize_qkv_e4m3(const void* q, const void* k, const void* v, void* q8, void* k8,
                         void* vt8, float* descale_q, float* descale_k, float* descale_v, int B,
                         int H, int N, int d, void* stream);

/*
 * fa_fwd_e4m3 — the forward of fa_fwd on E4M3 codes:
 *   q8, k8    : device, E4M3 codes [B, H, N, d], 16-byte aligned.
 *   vt8       : device, E4M3 codes of V keys-last [B, H, d, P] (P = N
 *               rounded up to 16), 16-byte aligned; columns >= N are ignored.
 *   descale_q, descale_k, descale_v : device, fp32 [B, H], 4-byte aligned.
 *   o, lse    : as for fa_fwd (bf16 O, fp32 L in natural-log units of the
 *               scaled scores of the dequantised Q and K).
 *   d         : 64 or 128.  causal, stream: as for fa_fwd.  scale: finite
 *               and >= 0 (negative: FA_ERR_UNSUPPORTED).
 * Errors: as for fa_fwd; d not 64 or 128: FA_ERR_UNSUPPORTED; a NULL descale:
 * FA_ERR_INVALID_ARG; o or lse overlapping any input: FA_ERR_INVALID_ARG.
 * Enqueues one kernel.
 */
int fa_fwd_e4m3(const void* q8, const void* k8, const void* vt8, const float* descale_q,
                const float* descale_k, const float* descale_v, void* o, float* lse, int B,
                int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_attn_unfused — standard attention in three steps with S and P in
 * device memory, the computation the fused forward replaces, kept as its
 * IO-awareness measurement ("How FlashAttention got past the O(N^2) memory
 * wall", "The standard-attention bottleneck: O(N^2) HBM round trips",
 * Steps 1-4; "Before implementing FlashAttention in Triton: FA1, 2 forward
 * pass", "Why it is needed"):
 *   1. S = scale Q K^T          fp32 [B*H][N][Np] in `workspace`
 *   2. L = ln sum_k exp(S_ik), P = exp(S - L)   (P bf16 [B*H][N][Np])
 *   3. O = P V                  bf16
 * with Np = N rounded up to 8.  Under the causal mask, S is computed only for
 * tiles that hold a visible key, step 2 reads only visible keys and writes P
 * (zeros at masked keys) up to the end of each row's 128-row tile, and step
 * 3 reads P and V only up to there.  Same O and L as fa_fwd, up to rounding
 * (S is fp32, P is bf16 and normalised before the product).
 *
 *   q, k, v, o, lse, B, H, N, d, scale, causal, stream: as for fa_fwd (any
 *               finite scale).
 *   workspace : device memory owned by the caller, 16-byte aligned, at least
 *               fa_attn_unfused_workspace_size(B, H, N, d) bytes, not
 *               overlapping q, k, v, o or lse.  Layout: S fp32
 *               [B*H][N][Np], padded to a multiple of 256 bytes, then P bf16
 *               [B*H][N][Np].  Contents on entry are ignored; on return S
 *               holds the scores of the computed tiles and P the
 *               probabilities (columns >= N and skipped tiles undefined).
 *   workspace_bytes : its size.
 * Errors: as for fa_fwd; a missing, too small or overlapping workspace:
 * FA_ERR_INVALID_ARG; an unaligned one: FA_ERR_MISALIGNED; sizes whose S and
 * P exceed 2^44 elements: FA_ERR_UNSUPPORTED.  Enqueues three kernels.
 */
int fa_attn_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int N, int d, float scale, int causal, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * Workspace bytes of fa_attn_unfused: round_up(B*H*N*Np*4, 256) + B*H*N*Np*2
 * with Np = N rounded up to 8.  0 if an argument is out of range.
 */
size_t fa_attn_unfused_workspace_size(int B, int H, int N, int d);

/*
 * fa_check_errors — synchronise `stream`, then report and clear the device
 * error record: FA_ERR_TIMEOUT if a bounded wait expired in any kernel since
 * the last check (the outputs of that call are then invalid), FA_ERR_CUDA if
 * the synchronisation failed, else FA_OK.
 */
int fa_check_errors(void* stream);

/*
 * fa_selftest_wait_timeout — exercise the failure path of the kernels'
 * bounded waits: enqueues one kernel whose single warp waits on a barrier
 * that nothing ever arrives at.  The wait gives up after timeout_us
 * microseconds (1 .. 1,000,000) and records the site (901) in the device
 * error record, so the next fa_check_errors returns FA_ERR_TIMEOUT and
 * fa_get_last_error_record reports {1, 901, 0, 0}.  Nothing faults or
 * hangs; the context stays usable.  Errors: timeout_us out of range:
 * FA_ERR_INVALID_ARG.
 */
int fa_selftest_wait_timeout(unsigned int timeout_us, void* stream);

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
