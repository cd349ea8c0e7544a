/*
 * oa.h -- C ABI of the online-softmax tiled attention library for GB300
 * (sm_103a).  Plain pointers and sizes only; no C++ or framework types.
 *
 * What it computes (sources are web pages on online softmax):
 *   - "Online Softmax -- the mathematical heart of FlashAttention"
 *     (inference-engineering roadmap page): s.1 three-pass safe softmax,
 *     s.2 online recurrence, s.4 tile recurrence, s.5 attention promotion,
 *     s.7 numerics (fp32 accumulation, fully masked rows).
 *   - "Online Softmax" (research-hub concept page), "Key math": running
 *     (m, l, o) with rescale alpha = exp(m_old - m_new), exact result.
 *   - "Online softmax in attention -- why and how": scores
 *     (q . k) / sqrt(hd), causal mask t2 <= t1 (positions along the
 *     sequence; with Nq queries and Nk keys the queries are the sequence's
 *     last Nq positions, so key j is visible to query i iff
 *     j <= i + (Nk - Nq)).
 *   - "Online Softmax & FlashAttention -- AI infra interview lesson":
 *     Step 1 (m, l) merge with the both-sides -inf special case and
 *     LSE = m + log l; Step 2 normalised-output merge; Steps 3-5
 *     (Q-outer order returning LSE, causal tile classes, split-KV decode
 *     merged by LSE).
 *
 * Conventions shared by every entry point
 *   Ownership   The caller owns every buffer.  All data pointers are DEVICE
 *               pointers (cudaMalloc / framework allocations) unless stated.
 *               The library allocates no device memory.
 *   Streams     Every compute call is asynchronous on `stream` (a
 *               cudaStream_t; NULL means the legacy default stream).  A
 *               successful return means the work was enqueued.
 *   Errors      Arguments are validated on the host before anything is
 *               launched; an invalid call launches nothing and returns
 *               OA_ERR_INVALID or OA_ERR_UNSUPPORTED.  A failed launch
 *               returns OA_ERR_CUDA.  Kernels never trap: every wait on the
 *               device is bounded, and a wait that expires records a code in
 *               a device status word, after which the kernel tears down and
 *               returns.  oa_sync_status() reports (and clears) that word.
 *               oa_last_error() gives a one-line description of the most
 *               recent failure on the calling thread.
 *   Masking     -inf scores/inputs contribute exactly zero.  A row with no
 *               visible element (all -inf, kv_len 0, or an empty split) has
 *               output +0.0 and LSE -inf; no path produces NaN.
 *   LSE         Natural-log log-sum-exp of the (scaled) scores of the row.
 */
#ifndef OA_H_
#define OA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* oa_stream_t;

typedef enum {
  OA_OK = 0,
  OA_ERR_INVALID = 1,     /* bad pointer, size, stride or alignment */
  OA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
  OA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
  OA_ERR_TIMEOUT = 4      /* a bounded device wait expired (see oa_sync_status) */
} oa_status;

typedef enum { OA_F32 = 0, OA_BF16 = 1 } oa_dtype;

/* Static text for a status code. */
const char* oa_status_string(int status);

/* One-line description of the last failure on the calling thread ("" if none). */
const char* oa_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int oa_version(void);

/*
 * Row softmax with per-row log-sum-exp.
 *   y[r, j] = exp(x[r, j] - m_r) / l_r,  lse[r] = m_r + ln l_r,
 *   m_r = max_j x[r, j],  l_r = sum_j exp(x[r, j] - m_r),
 * computed in one read of x: per-thread running (m, l) (roadmap page s.2),
 * merged across threads, warps and the CTAs of a cluster with the (m, l)
 * merge (interview lesson Step 1).  Rows wider than the on-chip capacity
 * (65536 fp32) are streamed twice instead of once.
 *   x      fp32 [rows, cols], row stride ld_x elements (ld_x >= cols).
 *   y      fp32 [rows, cols], row stride ld_y (ld_y >= cols), or NULL for
 *          statistics only.  y may be x itself (same pointer and stride);
 *          any other overlap is undefined.
 *   lse    fp32 [rows], or NULL.  y and lse may not both be NULL.
 * A fully -inf row gives y = +0.0 and lse = -inf.  Inputs must be finite
 * or -inf (+inf and NaN are outside the contract).
 * Errors: OA_ERR_INVALID for NULL x, rows or cols < 1, a stride < cols or
 * both outputs NULL.
 */
oa_status oa_softmax_rows(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y,
                          int64_t ld_y, float* lse, oa_stream_t stream);

/*
 * Fused attention forward, O = softmax(Q K^T * scale) V, with per-row LSE,
 * never writing the Nq x Nk score matrix to memory (roadmap page s.5;
 * interview lesson Step 3: Q-outer loop, one normalisation at the end,
 * LSE returned; Step 4: causal tiles skipped, fully visible or masked).
 *   q      [B, H, Nq, d], k and v [B, H, Nk, d], o [B, H, Nq, d]: all of
 *          dtype dt, contiguous row-major, 16-byte aligned.
 *   lse    fp32 [B, H, Nq], or NULL.
 *   causal 0 or 1.  The Nq queries are the last Nq positions of the Nk
 *          keys' sequence (new tokens after a KV cache of Nk - Nq keys:
 *          chunked prefill, multi-token decode), so key j is visible to
 *          query i iff j <= i + (Nk - Nq); j <= i when Nq == Nk.  With
 *          Nq > Nk the first Nq - Nk queries see no key (O = +0.0, LSE =
 *          -inf).  kv_len masks keys on top of this; it does not move the
 *          diagonal.
 *   scale  multiplies q . k before the softmax (callers normally pass
 *          1/sqrt(d)).  Must be finite and > 0.
 *   kv_len NULL, or a device int32 [B]: keys j >= kv_len[b] are masked
 *          (values are clamped to [0, Nk]).
 * bf16: tcgen05 tensor-core kernel, fp32 accumulation, bf16 O; d must be
 * 64 or 128 (else OA_ERR_UNSUPPORTED).  fp32: SIMT kernel in fp32,
 * 1 <= d <= 256.
 * Results are deterministic for a given shape and device.  A causal row's
 * key tiles are summed in an order that follows how the launch deals its
 * work to the SMs, so devices with different SM counts may differ in the
 * last bits (within the stated tolerances).
 * Errors: OA_ERR_INVALID for NULL q/k/v/o, sizes < 1 (B, H, Nq, Nk, d),
 * misalignment or a bad scale; OA_ERR_UNSUPPORTED for an unsupported
 * (dtype, d).
 */
oa_status oa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt,
                      int B, int H, int Nq, int Nk, int d, int causal, float scale,
                      const int32_t* kv_len, oa_stream_t stream);

/*
 * oa_attn_fwd with grouped key/value heads: k and v are [B, H_kv, Nk, d]
 * and query head h reads key/value head h / (H / H_kv).  H_kv == H is
 * oa_attn_fwd.  The pages' attention has one key/value head per query head;
 * the grouping is the library generalisation that the interview lesson's
 * "In Real Systems" list of library entry points (fixed-length, variable-
 * length and KV-cache calls) is read to ask for.
 *   q, o [B, H, Nq, d]; k, v [B, H_kv, Nk, d]; everything else as in
 *   oa_attn_fwd (dtype, alignment, lse, causal, scale, kv_len, support).
 * Decode (bf16, d = 64 / 128, (H / H_kv) * Nq <= 128: one or a few new
 * tokens per sequence): the query heads of a group hold (H / H_kv) * Nq
 * consecutive rows of q, o and lse, which run as the rows of one
 * [B, H_kv, (H / H_kv) * Nq, d] problem, so each group's K/V is read once;
 * causal positions are taken per query token (a row's index modulo Nq).
 * One query with causal set sees every key and runs as non-causal.
 * Errors: those of oa_attn_fwd, plus OA_ERR_INVALID when H_kv < 1 or
 * H_kv does not divide H.
 */
oa_status oa_attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                          oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d, int causal,
                          float scale, const int32_t* kv_len, oa_stream_t stream);

/*
 * Fused attention forward over packed sequences of different lengths (the
 * variable-length entry point of the interview lesson's "In Real Systems"
 * list), tcgen05 tensor-core kernel.  Sequence s owns query tokens
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key tokens
 * [cu_seqlens_k[s], cu_seqlens_k[s+1]); each is attended independently,
 * exactly as oa_attn_fwd does for one (b, h).
 *   q, o    bf16 [total_q, H, d] (token-major), 16-byte aligned.
 *   k, v    bf16 [total_k, H_kv, d]; query head h reads head h / (H/H_kv).
 *   lse     fp32 [total_q, H], or NULL.
 *   cu_seqlens_q, cu_seqlens_k   device int32 [num_seqs + 1], non-decreasing;
 *           entries are clamped to [0, total].  A sequence with no keys gets
 *           O = 0 and lse = -inf; one with no queries writes nothing.
 *   max_seqlen_q, max_seqlen_k   the longest query / key sequence.  A
 *           query sequence longer than max_seqlen_q has its tail rows left
 *           unwritten and the status word records it (oa_sync_status).
 *   causal  0 or 1: a sequence with lq queries and lk keys has its queries
 *           at its last lq positions, so its key j is visible to its query
 *           i iff j <= i + (lk - lq) (j <= i for equal lengths).
 *   d       64 or 128.
 * The caller keeps every buffer alive until the work has completed on
 * `stream`; nothing is allocated.  As for oa_attn_fwd, results are
 * deterministic for given inputs and device; a causal row's key tiles are
 * summed in an order that follows the launch's dealing, which the kernel
 * chooses from the sequence lengths, so the last bits may differ between
 * devices with different SM counts.
 * Errors: OA_ERR_INVALID (NULL pointers, sizes, alignment, H_kv not
 * dividing H, bad scale); OA_ERR_UNSUPPORTED (dtype other than bf16, d).
 */
oa_status oa_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             oa_dtype dt, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, int num_seqs, int H, int H_kv,
                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                             int causal, float scale, oa_stream_t stream);

/*
 * Bytes of device workspace oa_attn_fwd_host needs: device copies of q, k,
 * v, o (dtype dt) and lse (fp32), each rounded up to 256 bytes.  0 for
 * invalid arguments.
 */
size_t oa_attn_fwd_host_workspace_bytes(oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d);

/*
 * oa_attn_fwd_gqa on HOST buffers: copies q, k, v in, runs the forward and
 * copies o and lse back, overlapping the three.  A library addition with no
 * counterpart on the source pages, for callers whose tensors live in host
 * memory (the whole call is what a host-side user pays).  The B * H_kv
 * key/value planes are cut into `chunks` pieces (0: the library's default of
 * 4) whose sizes fall linearly, so that little work follows the last copy
 * in; the copy in of piece c + 1, the kernel of piece c and the copy out of
 * piece c - 1 run at the same time on three streams the library keeps for
 * each device (created on the first call on that device; make that call
 * before any stream capture).  The result equals that of oa_attn_fwd_gqa
 * on the whole batch bit for bit (each piece sums its key tiles in the
 * whole call's order).
 *   q_host, k_host, v_host, o_host, lse_host: host memory in the layouts of
 *          oa_attn_fwd_gqa (lse_host may be NULL), 16-byte aligned.  For the
 *          copies to overlap they must be page-locked (cudaHostAlloc,
 *          pinned); they must stay valid, and the inputs unchanged, until
 *          the call's work has completed on `stream`.
 *   workspace: device memory of >= oa_attn_fwd_host_workspace_bytes(...)
 *          bytes, 256-byte aligned, owned by the caller.
 *   chunks: 0 .. 64.  kv_len is not supported here (all keys visible).
 * Ordering: the work starts after everything queued on `stream` before the
 * call and `stream` waits for all of it, so a synchronisation of `stream`
 * covers the outputs.  Calls on one device are serialised by the library
 * (they share its streams).
 * Errors: those of oa_attn_fwd_gqa (checked before anything is queued), plus
 * OA_ERR_INVALID for a bad chunks value or workspace.  A CUDA error after
 * some pieces were queued returns OA_ERR_CUDA; the queued work still runs.
 */
oa_status oa_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                           float* lse_host, oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d,
                           int causal, float scale, int chunks, void* workspace, size_t workspace_bytes,
                           oa_stream_t stream);

/*
 * The fp32 SIMT attention forward with explicit tile sizes: Br query rows
 * per CTA and Bc keys per step of the online recurrence (1 <= Br, Bc <= 64).
 * Same contract as oa_attn_fwd with dt = OA_F32; the result does not
 * depend on the tiles beyond rounding.  Follows the lesson's worked shapes
 * (Br = 4, Bc = 3) when asked to.
 */
oa_status oa_attn_fwd_f32_tiles(const float* q, const float* k, const float* v, float* o,
                                float* lse, int B, int H, int Nq, int Nk, int d, int causal,
                                float scale, const int32_t* kv_len, int Br, int Bc,
                                oa_stream_t stream);

/*
 * Bytes of workspace oa_attn_bwd needs: B*H*Nq * (d + 1) fp32 values (the
 * fp32 dQ accumulator, then D = rowsum(dO * O)), rounded up to 256 bytes.
 * 0 for invalid sizes.
 */
size_t oa_attn_bwd_workspace_bytes(int B, int H, int Nq, int d);

/*
 * Fused attention backward (tcgen05 tensor-core kernel): the gradients
 * dQ, dK, dV of O = softmax(Q K^T * scale) V for a given dO, with the
 * probabilities recomputed tile by tile from the forward's per-row LSE
 * instead of read back (page "Online softmax in attention -- why and how",
 * section "Where this is heading: FA2": on backward, the scores are
 * recomputed from the cached running max and sum, which the LSE folds into
 * one number).  The Nq x Nk matrices P and dP never reach memory.  Three
 * launches on `stream`: D = rowsum(dO * O) (and zeroing of the dQ
 * accumulator), one CTA per 128-key tile of each (b, h) that accumulates
 * dK and dV on chip and adds its dQ share to the fp32 accumulator, and the
 * dQ conversion to bf16.
 *   q, o, dout, dq  bf16 [B, H, Nq, d]; k, v, dk, dv  bf16 [B, H, Nk, d];
 *           contiguous row-major, 16-byte aligned.  o and lse are the
 *           forward's outputs for the same q, k, v, causal and scale.
 *   lse     fp32 [B, H, Nq], non-NULL.  A row with lse = -inf (no visible
 *           key) gets dQ = 0 and contributes nothing to dK, dV.
 *   causal  0 or 1 (key j visible to query i iff j <= i + (Nk - Nq), as in
 *           oa_attn_fwd).
 *   scale   finite and > 0.
 *   d       64 or 128.
 *   workspace  device, >= oa_attn_bwd_workspace_bytes(B, H, Nq, d) bytes,
 *           16-byte aligned; owned by the caller, who must not touch it (or
 *           dq, dk, dv) until the call's work has completed on `stream`.
 *           Its contents on entry do not matter.
 * dK and dV are written with plain stores, one CTA per key tile, so the
 * result is deterministic; dQ sums fp32 atomics and may differ in the last
 * bits from run to run.
 * Errors: OA_ERR_INVALID (NULL pointers, sizes < 1, misalignment, a bad
 * scale, workspace too small); OA_ERR_UNSUPPORTED (dtype other than bf16,
 * d other than 64 / 128).
 */
oa_status oa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, oa_dtype dt, int B, int H,
                      int Nq, int Nk, int d, int causal, float scale, void* workspace,
                      size_t workspace_bytes, oa_stream_t stream);

/*
 * oa_attn_bwd with grouped key/value heads: k, v, dk, dv are [B, H_kv, Nk, d]
 * and query head h reads key/value head h / (H / H_kv), as in
 * oa_attn_fwd_gqa.  dK and dV of a key/value head sum the contributions of
 * every query head of its group: one CTA per 128 keys of a key/value head
 * steps through all query tiles of all the group's heads, so the sums stay
 * on chip (no atomics) and remain deterministic.  H_kv == H is oa_attn_bwd.
 * Same workspace (oa_attn_bwd_workspace_bytes(B, H, Nq, d)), support and
 * errors as oa_attn_bwd, plus OA_ERR_INVALID when H_kv < 1 or does not
 * divide H.
 */
oa_status oa_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, oa_dtype dt, int B, int H,
                          int H_kv, int Nq, int Nk, int d, int causal, float scale, void* workspace,
                          size_t workspace_bytes, oa_stream_t stream);

/*
 * oa_attn_bwd over packed sequences of different lengths (the gradients of
 * oa_attn_fwd_varlen): sequence s owns query tokens [cu_seqlens_q[s],
 * cu_seqlens_q[s+1]) and key tokens [cu_seqlens_k[s], cu_seqlens_k[s+1]),
 * each differentiated on its own, with grouped key/value heads as in
 * oa_attn_bwd_gqa.
 *   q, o, dout, dq  bf16 [total_q, H, d] (token-major), 16-byte aligned.
 *   k, v, dk, dv    bf16 [total_k, H_kv, d].
 *   lse     fp32 [total_q, H] from oa_attn_fwd_varlen on the same inputs.
 *   cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k: as in
 *           oa_attn_fwd_varlen.  One CTA per 128 keys up to max_seqlen_k
 *           of each (sequence, key/value head); a key sequence longer than
 *           max_seqlen_k has its tail keys' dK, dV left unwritten and the
 *           status word records it (oa_sync_status returns
 *           OA_ERR_INVALID).  max_seqlen_q is accepted for symmetry with the
 *           forward and not needed.  Keys that no query sees get dK = dV = 0;
 *           queries of a sequence without keys get dQ = 0.
 *   workspace: >= oa_attn_bwd_workspace_bytes(1, H, total_q, d) bytes.
 * Errors: those of oa_attn_bwd_gqa, plus OA_ERR_INVALID for NULL or
 * misaligned cu_seqlens, num_seqs < 1 or max_seqlen_k outside
 * [1, total_k].
 */
oa_status oa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             oa_dtype dt, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int num_seqs, int H, int H_kv, int total_q, int total_k,
                             int max_seqlen_q, int max_seqlen_k, int d, int causal, float scale,
                             void* workspace, size_t workspace_bytes, oa_stream_t stream);

/*
 * Bytes of workspace oa_attn_splitkv needs: num_splits * B*H*Nq * (d + 1)
 * fp32 values (normalised partial outputs, then their LSEs), rounded up to
 * 256 bytes.  0 for invalid sizes.
 */
size_t oa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * Split-KV attention (decode style; interview lesson Step 5): the keys of
 * each row are cut into num_splits chunks of ceil(Nk / num_splits); one
 * CTA per (row, chunk) runs the online recurrence over its chunk and writes
 * the chunk's normalised output O_c and lse_c (an empty chunk writes
 * O_c = 0, lse_c = -inf); a second kernel merges the partials with the LSE
 * merge of oa_lse_merge.  Non-causal.
 *   q [B, H, Nq, d], k and v [B, H, Nk, d], o [B, H, Nq, d]: dtype dt,
 *   contiguous, 16-byte aligned.  lse fp32 [B, H, Nq] or NULL.
 *   kv_len NULL or device int32 [B] (clamped to [0, Nk]).
 *   workspace: device, >= oa_splitkv_workspace_bytes(...) bytes, 16-byte
 *   aligned; the caller owns it and must not touch it until the call's
 *   work has completed on `stream`.
 * Supported: bf16 with d in {8, 16, 32, 64, 128, 256}; fp32 with d in
 * {4, 8, 16, 32, 64, 128}; 1 <= num_splits <= 1024.
 * Errors: OA_ERR_INVALID (NULL, sizes, alignment, workspace too small),
 * OA_ERR_UNSUPPORTED (dtype/d).
 */
oa_status oa_attn_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                          oa_dtype dt, int B, int H, int Nq, int Nk, int d, float scale,
                          const int32_t* kv_len, int num_splits, void* workspace,
                          size_t workspace_bytes, oa_stream_t stream);

/*
 * oa_attn_splitkv with grouped key/value heads (KV-cache decode with fewer
 * key/value heads than query heads): k and v are [B, H_kv, Nk, d] and query
 * head h reads head h / (H / H_kv); kv_len gives each sequence's cache
 * length.  Same workspace size and support matrix as oa_attn_splitkv.
 * Grouped decode takes no split: with bf16, d = 64 / 128 and
 * (H / H_kv) * Nq <= 128, the group's query heads x queries are
 * consecutive rows of q, o and lse and are computed together by the
 * tensor-core forward kernel (one launch), every K/V row read once for the
 * whole group.  On that path num_splits and the workspace are checked but
 * NOT USED; the result is the same attention.  Other grouped calls (more
 * rows per group, fp32) split the keys into num_splits chunks and merge, as
 * oa_attn_splitkv does.
 * Errors: those of oa_attn_splitkv, plus OA_ERR_INVALID when H_kv < 1 or
 * H_kv does not divide H.
 */
oa_status oa_attn_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                              oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d,
                              float scale, const int32_t* kv_len, int num_splits, void* workspace,
                              size_t workspace_bytes, oa_stream_t stream);

/*
 * Split-KV attention that allocates nothing -- a library addition with no
 * counterpart on the source pages.  Same arguments, result and support
 * matrix as oa_attn_splitkv, minus the workspace: the partials live in one
 * 16 MiB scratch array built into the library (held on every GPU that
 * loads the library, until the process exits).  For callers that cannot
 * allocate device memory when they call -- code inside a host application
 * that owns all device memory through its own allocator, or a
 * latency-critical path where an allocation could block or fail.
 *   Limit: num_splits * B*H*Nq * (d + 1) * 4 bytes <= 16 MiB; larger
 *          requests return OA_ERR_INVALID and launch nothing.
 *   Set-up: the first call on a device looks up the array's device address
 *          (cudaGetSymbolAddress) with that device current.  Under CUDA's
 *          default lazy module loading that lookup also loads the module
 *          holding the array and commits its 16 MiB on that device, so the
 *          first call is the only one that can fail for lack of device
 *          memory (OA_ERR_CUDA) or wait on the driver: make one call with
 *          valid arguments at start-up, before the latency-critical path
 *          and before any stream capture.
 *   Sharing: every call uses the same array.  Calls whose work overlaps on
 *          the GPU (other streams, other host threads) race on it; the
 *          caller must serialise them.  Nothing in the array needs to start
 *          at zero: each call writes every partial it reads.
 */
oa_status oa_attn_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                 oa_dtype dt, int B, int H, int Nq, int Nk, int d, float scale,
                                 const int32_t* kv_len, int num_splits, oa_stream_t stream);

/*
 * Merge of S split partials per row (interview lesson Step 1 merge and
 * Step 2 normalised-output rule; log-sum-exp form):
 *   L = max_c lse_c,  w_c = exp(lse_c - L),  W = sum_c w_c,
 *   lse = L + ln W,   o = sum_c (w_c / W) o_c,
 * with o = +0.0 and lse = -inf when every lse_c is -inf.
 *   part_o   fp32 [S, R, d] normalised partial outputs, or NULL iff d == 0.
 *   part_lse fp32 [S, R].
 *   o        [R, d] of dtype o_dt (fp32 or bf16), or NULL iff d == 0.
 *   lse      fp32 [R], or NULL (then d must be > 0).
 * Alignment: part_o and o 16-byte aligned when d % 4 == 0 (vector path);
 * any 4-byte alignment otherwise.  1 <= S <= 65535, R >= 1, 0 <= d <= 1024.
 */
oa_status oa_lse_merge(const float* part_o, const float* part_lse, int S, int64_t R, int d,
                       void* o, oa_dtype o_dt, float* lse, oa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word that
 * kernels set when a bounded wait expires.  Returns OA_OK, OA_ERR_TIMEOUT
 * (with the code of the expired wait in oa_last_error()), OA_ERR_INVALID
 * when oa_attn_fwd_varlen met a query sequence longer than its
 * max_seqlen_q, or OA_ERR_CUDA if the synchronisation itself failed.
 */
oa_status oa_sync_status(oa_stream_t stream);

/*
 * Upper bound, in nanoseconds, on any single device-side wait (default
 * 2e9).  Applies to launches made after the call.  0 restores the default.
 */
void oa_set_wait_limit_ns(uint64_t ns);

/*
 * Self-test of the failure path: launches one warp that waits, with the
 * library's bounded wait, on an mbarrier that nothing ever arrives on.  The
 * wait gives up after `limit_ns` nanoseconds and records a timeout in the
 * status word; oa_sync_status() then returns OA_ERR_TIMEOUT and the context
 * stays usable.  limit_ns must be in [1e3, 1e10].
 */
oa_status oa_selftest_wait_timeout(uint64_t limit_ns, oa_stream_t stream);

/*
 * Self-test of the debug build's checks: launches one warp whose single
 * store of 1 to the device int `flag` is guarded by a check that fails.  In
 * the debug build (the library compiled with -DOA_DEBUG, liboa_debug.so) the
 * check records its site in the status word and skips the store, so *flag is
 * left as it was and oa_sync_status() returns OA_ERR_INVALID; in the release
 * build checks are compiled out, the store happens and oa_sync_status()
 * returns OA_OK.  flag: device pointer to one int, 4-byte aligned.  Errors:
 * OA_ERR_INVALID for a NULL or misaligned flag.
 */
oa_status oa_selftest_debug_check(int* flag, oa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OA_H_ */
