/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused attention forward library
 * (libfa_gb300.so).
 *
 * The operation is scaled-dot-product attention, forward pass, with the
 * log-sum-exp of every row:
 *
 *     S = scale * Q K^T             (per batch b and head h; N x N scores)
 *     S[i][j] = -inf  for j > i     (causal only: query i sees keys 0..i)
 *     LSE[i]  = ln sum_j exp(S[i][j])
 *     O[i]    = sum_j exp(S[i][j] - LSE[i]) V[j]
 *
 * Sources: LeetCUDA "flash_attn_mma_tiling_qk.cu" (the FlashAttention-2
 * forward: Q,K,V,O as [batch, heads, seq_len, head_dim]; scores scaled before
 * the exponential; the online row max / row sum recurrence and the final
 * division by the row sum); flash-attention "hopper/flash_fwd_kernel.h"
 * (persistent warp-specialised forward that stores O together with the row
 * log-sum-exp; an empty row stores O = 0, LSE = -inf) and
 * "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp" (the causal mask and the meaning
 * of the stored LSE: the log-normaliser of the scaled scores, consumed by the
 * backward pass as exp2(S*scale_log2 - LSE_log2)).  The LSE written here is in
 * natural-log units.
 *
 * All entry points are plain C: pointers and sizes, no C++ or framework types,
 * no exceptions.  Every function returns an fa_status_t code (or a string).
 *
 * Launches: every kernel is launched with programmatic stream serialisation
 * (programmatic dependent launch).  It may begin its set-up while the
 * previous kernel of the stream finishes, but reads and writes global memory
 * only after that kernel has completed; stream order is therefore unchanged
 * for the caller.  A caller's own kernel launched the same way right after
 * one of these must wait (griddepcontrol.wait) before using its results, as
 * with any programmatic dependent launch.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>

/* Exported from the shared library (built with hidden default visibility). */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and o. */
typedef enum {
  FA_DTYPE_F16 = 0,  /* IEEE binary16 */
  FA_DTYPE_BF16 = 1  /* bfloat16 */
} fa_dtype_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad flag/scale */
  FA_ERR_UNSUPPORTED = 2,     /* head dim / device not supported */
  FA_ERR_MISALIGNED = 3,      /* a pointer breaks the alignment rule below */
  FA_ERR_CUDA = 4,            /* a CUDA runtime call or the launch failed */
  FA_ERR_DEVICE_TIMEOUT = 5,  /* a device-side wait ran out (watchdog) */
  FA_ERR_SCRATCH_LIMIT = 6    /* the split partials would not fit in the
                                 library's fixed scratch (fa_fwd_splitkv_noalloc) */
} fa_status_t;

/*
 * fa_fwd -- attention forward pass on the current CUDA device.
 *
 * Arguments
 *   q, k, v  device pointers, each a contiguous row-major [B][H][N][d] tensor
 *            of `dtype` (the layout of the LeetCUDA kernel's Q,K,V).
 *   o        device pointer, contiguous [B][H][N][d] of `dtype`; written.
 *   lse      device pointer, contiguous [B][H][N] float32 (natural-log
 *            log-sum-exp of the scaled scores of each row); written.  May be
 *            NULL, in which case no LSE is stored.
 *   B, H, N  batch, heads, sequence length.  Any of them 0: nothing is done
 *            and FA_OK is returned (pointers are not touched).  Negative:
 *            FA_ERR_INVALID_ARG.  B*H must be < 2^31 and N < 2^31.
 *   d        head dimension: 64, 128 or 256 (other values: FA_ERR_UNSUPPORTED).
 *   scale    softmax scale applied to Q.K^T; must be finite and > 0
 *            (1/sqrt(d) is the usual choice).
 *   causal   0: every query sees every key; 1: query i sees keys 0..i.
 *   dtype    fa_dtype_t.
 *   stream   a cudaStream_t (NULL: the legacy default stream).
 *
 * Alignment: q, k, v, o must be 16-byte aligned; lse 4-byte aligned
 * (else FA_ERR_MISALIGNED).  Ownership: the caller owns every buffer; the
 * call allocates no device memory.  The call enqueues one kernel on `stream`
 * and returns without synchronising; argument errors are reported before
 * anything is enqueued; a launch failure returns FA_ERR_CUDA.  A device-side
 * wait that runs out (a hung pipeline) is reported later by
 * fa_get_device_status().  Requires an sm_103 GPU (else FA_ERR_UNSUPPORTED).
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, int dtype,
           void* stream);

/*
 * fa_fwd_ext -- fa_fwd with grouped K/V heads and a local window.
 *
 * Sources: flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp", the
 * qhead_per_khead (grouped-query / multi-query attention) and
 * window_size_left / window_size_right (local attention, its Is_local mask)
 * options of CollectiveMainloopBwd.
 *
 *   k, v     contiguous [B][H_kv][N][d]; query head h (of H) reads K/V head
 *            h / (H / H_kv).  H must be a multiple of H_kv (else
 *            FA_ERR_INVALID_ARG); H_kv = H is ordinary multi-head attention,
 *            H_kv = 1 multi-query attention.
 *   window_left, window_right
 *            query i sees keys j with i - window_left <= j <= i + window_right;
 *            a negative value leaves that side unbounded.  With causal = 1 the
 *            right bound is 0 whatever window_right says.  Every row sees at
 *            least its own key, so no row is empty.
 * All other arguments, the layout of q, o, lse, alignment, ownership and
 * error behaviour are those of fa_fwd (which is fa_fwd_ext with H_kv = H and
 * both window bounds -1).
 */
FA_API int fa_fwd_ext(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int H_kv, int N, int d, float scale, int causal,
                      int window_left, int window_right, int dtype, void* stream);

/*
 * fa_fwd_varlen -- fa_fwd_ext over a batch of sequences of different
 * lengths packed along the rows (self-attention: each sequence's queries
 * attend to that sequence's keys only).
 *
 * Source: flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp" and the
 * older "hopper/flash_fwd_kernel.h" (their variable-length mode: cu_seqlens
 * row offsets into packed tensors, per-sequence lengths through
 * seqlen_traits, and the tile loops bounded by each sequence's own length).
 *
 *   q, o        device pointers, contiguous [total][H][d] of `dtype`.
 *   k, v        contiguous [total][H_kv][d]; grouped heads as in fa_fwd_ext.
 *   lse         contiguous [H][total] float32, or NULL.
 *   cu_seqlens  device pointer to batch + 1 int32 row offsets, 4-byte
 *               aligned: sequence b is rows [cu_seqlens[b], cu_seqlens[b+1]).
 *               They must be non-decreasing, within [0, total], and no
 *               sequence longer than max_seqlen; the kernels clamp offsets
 *               and lengths to those bounds, so a malformed array can only
 *               leave rows unwritten, never touch memory outside the tensors.
 *               Rows outside every sequence are not written.  The offsets are
 *               absolute row indices, so a pointer into a longer offset array
 *               (with batch counting from there) runs a subset of consecutive
 *               sequences alone, writing exactly their rows, bit for bit as
 *               the call over all of them would.
 *   batch, max_seqlen, total
 *               number of sequences, the longest length, and the packed row
 *               count; any of them 0: nothing is done (FA_OK).  Negative:
 *               FA_ERR_INVALID_ARG.
 *   causal, window_left, window_right
 *               as in fa_fwd_ext, with positions counted from the start of
 *               each sequence.
 * The last query tile of a sequence reads up to 127 rows of the following
 * sequence as padding (masked out): the packed tensors must hold finite
 * values.  Alignment, ownership, scale, dtype and error behaviour are those
 * of fa_fwd.
 */
FA_API int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                         const int* cu_seqlens, int batch, int max_seqlen, int total, int H,
                         int H_kv, int d, float scale, int causal, int window_left,
                         int window_right, int dtype, void* stream);

/*
 * fa_fwd_varlen_qk -- the variable-length forward with separate query and
 * key sequences: cross-attention, a prefill continuing a cached prefix, or
 * decoding a few query rows against a KV cache with spare capacity.
 *
 * Source: flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp"
 * (CollectiveMainloopBwd::Arguments: cu_seqlens_q, cu_seqlens_k,
 * seqused_k; get_seqlen_q / get_seqlen_k, which take a used length when one
 * is given and the offset difference otherwise; the causal and local masks
 * shifted by seqlen_k - seqlen_q) and the variable-length mode of
 * "hopper/flash_fwd_kernel.h" (rows without a key stored as O = 0,
 * LSE = -inf: store_zero).
 *
 *   q, o          contiguous [total_q][H][d] of `dtype`; lse [H][total_q]
 *                 float32 or NULL.
 *   k, v          contiguous [total_k][H_kv][d]; grouped heads as in
 *                 fa_fwd_ext.
 *   cu_seqlens_q, cu_seqlens_k
 *                 device pointers to batch + 1 int32 row offsets each
 *                 (4-byte aligned): sequence b owns query rows
 *                 [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key rows
 *                 [cu_seqlens_k[b], cu_seqlens_k[b+1]).  Passing one array for
 *                 both (with equal totals) is fa_fwd_varlen.
 *   seqused_q, seqused_k
 *                 NULL, or device pointers to batch int32 used lengths: only
 *                 the first seqused_q[b] query rows and seqused_k[b] key rows
 *                 of sequence b take part (a cache whose rows past the used
 *                 length hold anything).  Query rows past the used length are
 *                 not written.
 *   batch, max_seqlen_q, max_seqlen_k, total_q, total_k
 *                 sequence count, the longest used query and key lengths, and
 *                 the packed row counts.  batch, max_seqlen_q or total_q 0:
 *                 nothing is done (FA_OK).  max_seqlen_k or total_k 0 is
 *                 allowed: every query row then has no key.  Negative, or a
 *                 longest length of 2^30 or more: FA_ERR_INVALID_ARG.
 *   causal, window_left, window_right
 *                 bottom-right aligned: query i of a sequence with n_q used
 *                 queries and n_k used keys sits at key position
 *                 i + n_k - n_q, so causal keeps keys j <= i + n_k - n_q and
 *                 the window keeps i + n_k - n_q - window_left <= j <=
 *                 i + n_k - n_q + window_right (n_q = n_k: fa_fwd_varlen).
 *                 A query row with no admissible key gets O = 0 and
 *                 LSE = -inf.
 * Grouped query heads are packed into shared tiles (fa_set_gqa_pack).
 * Offsets and used lengths are clamped by the kernels to the packed tensors
 * and to max_seqlen_q / max_seqlen_k (a malformed array only shortens
 * sequences).  Tiles read up to 127 rows past a sequence's used rows (masked
 * out): the packed tensors must hold finite values.  Alignment, ownership,
 * scale, dtype and error behaviour are those of fa_fwd.
 */
FA_API int fa_fwd_varlen_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* seqused_q, const int* seqused_k, int batch,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                            int H, int H_kv, int d, float scale, int causal, int window_left,
                            int window_right, int dtype, void* stream);

/*
 * fa_fwd_splitkv -- fa_fwd_ext with the keys of every query row cut into
 * `num_splits` contiguous ranges that run as separate work units, then merged.
 *
 * Source: flash-attention "hopper/flash_fwd_kernel.h" (the older
 * FlashAttention-3 forward shell, compute_attn_ws): its work tiles carry a
 * key-split index (n_split_idx, Is_split) so that few (b,h) query tiles can
 * still fill the GPU.  The page stops at the split partials; the merge is
 * the log-sum-exp mixture of per-split softmaxes:
 *     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s,
 * where split s holds the row's admissible keys of its range (a split with
 * none of them is left out).
 *
 *   num_splits  requested split count; 0 picks one: 1 when the
 *               B*H*ceil(N/256) query units (ceil(N/128) per head for
 *               d = 256) are at least the SM count, else the count (up to 32)
 *               with the shortest estimated persistent-grid makespan.
 *               Clamped to the number of K/V tiles (128 keys; 64 for
 *               d = 256); the splits cover equal whole tiles, so the count
 *               used may be lower than asked.  Negative: FA_ERR_INVALID_ARG.
 *   workspace   device scratch of at least fa_splitkv_workspace_bytes()
 *               bytes for the same arguments, 256-byte
 *               aligned (else FA_ERR_MISALIGNED).  Layout: the 16-bit partial
 *               O of each split [S][B][H][N][d], then at the next 256-byte
 *               boundary the fp32 partial LSE [S][B][H][N].  Nothing in it
 *               needs to be initialised; it is overwritten.  May be NULL when
 *               the split count used is 1 (the call is then fa_fwd_ext).
 *   workspace_bytes  its size; smaller than required: FA_ERR_INVALID_ARG.
 *
 * The call enqueues two kernels on `stream` (the split forward, then the
 * merge); the workspace must not be used by another call until both ran.
 * O carries one more 16-bit rounding than fa_fwd_ext (of each partial).
 * Every other argument and rule is that of fa_fwd_ext; the call allocates
 * no device memory.
 */
FA_API int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int H_kv, int N, int d, float scale, int causal,
                          int window_left, int window_right, int dtype, int num_splits,
                          void* workspace, unsigned long long workspace_bytes,
                          void* stream);

/*
 * Workspace bytes fa_fwd_splitkv needs for these arguments (the same values
 * as its own; the split count chosen for num_splits = 0 depends on the mask
 * and on the current device's SM count), written to *bytes: 0 when the split
 * count used is 1 or the problem is empty.  Returns FA_OK, or
 * FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED for the argument errors of
 * fa_fwd_splitkv, FA_ERR_CUDA if the SM count cannot be read.
 */
FA_API int fa_splitkv_workspace_bytes(int B, int H, int N, int d, int causal,
                                      int window_left, int window_right, int num_splits,
                                      unsigned long long* bytes);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without a caller workspace: the
 * split partials go to a scratch array that the library keeps in static
 * device memory, FA_NOALLOC_SCRATCH_BYTES (32 MiB) per device.  The pages
 * have no counterpart: this entry point exists for callers that cannot
 * allocate at call time (no cudaMalloc / cudaFree, which can synchronise the
 * device, on a hot path; engines whose device memory is fixed at start-up;
 * plain C callers without a caching allocator).  The call allocates nothing,
 * through CUDA or any library.
 *
 *   num_splits  as for fa_fwd_splitkv, with the scratch as the workspace:
 *               an explicit count whose partials need more than
 *               FA_NOALLOC_SCRATCH_BYTES (fa_splitkv_workspace_bytes) is
 *               rejected with FA_ERR_SCRATCH_LIMIT before anything is
 *               enqueued; 0 takes the automatic count, lowered to the largest
 *               count whose partials fit.  A count that resolves to 1 split
 *               is the plain forward (no scratch used).
 *               S splits take S * B*H*N * (2d + 4) bytes (plus at most 255
 *               bytes of alignment), so at most
 *               floor(FA_NOALLOC_SCRATCH_BYTES / (B*H*N * (2d + 4))) fit:
 *               for example 3 for one head of 32768 rows at d = 128, where
 *               the automatic count of fa_fwd_splitkv without a mask is 7
 *               on a 152-SM GB300.  fa_splitkv_workspace_bytes with an explicit count
 *               tells whether that count fits.
 * Every other argument, layout, alignment rule and error is that of
 * fa_fwd_splitkv.
 *
 * Set-up: the first call on each device looks up that device's scratch
 * address (cudaGetSymbolAddress, which can load the library's device code),
 * and so does the first call after the device's context changed (a new
 * primary context after cudaDeviceReset, or a driver context the caller
 * made current); make that first call before capturing any stream.  A failed
 * look-up returns FA_ERR_CUDA, clears the runtime's last error and is retried
 * by the next call.
 *
 * Nothing in the scratch has to start at zero: each call writes every
 * partial it later reads.  All calls on one device share the one scratch, so
 * calls whose kernels may overlap (different streams without ordering
 * between them, or several host threads) race on it and can return wrong
 * results: order them on one stream or with events.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32ull << 20)

FA_API int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int H_kv, int N, int d,
                                  float scale, int causal, int window_left, int window_right,
                                  int dtype, int num_splits, void* stream);

/*
 * fa_fwd_fp8 -- attention forward on FP8 E4M3 inputs with descale factors.
 *
 * Source: flash-attention "hopper/flash_fwd_kernel.h" (its FP8 path:
 * E4M3 Q, K, V with descale_q/k/v, the Q K^T descales folded into the
 * softmax scale, P rounded to FP8 after an exponent offset ("Max_offset"),
 * V's descale applied to O, a 16-bit output).
 *
 *   q        device pointer, contiguous [B][H][N][d] E4M3 bytes.
 *   k, v     contiguous [B][H_kv][N][d] E4M3 bytes (grouped heads as in
 *            fa_fwd_ext).  The real inputs are descale_q * q, descale_k * k,
 *            descale_v * v (each factor finite and > 0).
 *   o        contiguous [B][H][N][d] bfloat16 (written).
 *   lse      [B][H][N] float32 natural-log LSE of the descaled scores, or NULL.
 *   d        128 (else FA_ERR_UNSUPPORTED).
 *   workspace  device scratch of at least fa_fwd_fp8_workspace_bytes()
 *            bytes, 256-byte aligned: receives V transposed
 *            ([B*H_kv][d][N rounded up to 128] bytes); need not be
 *            initialised.
 * P is rounded to E4M3 (3 mantissa bits) before the P V product: O carries
 * a relative error of up to 2^-4 of the V values it averages (typically far
 * less), while LSE is as accurate as in fa_fwd.  Enqueues two kernels (the V
 * transpose, the forward).  Other arguments, alignment and errors as in
 * fa_fwd_ext.
 */
FA_API int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int H_kv, int N, int d, float scale, float descale_q,
                      float descale_k, float descale_v, int causal, int window_left,
                      int window_right, void* workspace, unsigned long long workspace_bytes,
                      void* stream);

/* Workspace bytes of fa_fwd_fp8 for these sizes (written to *bytes). */
FA_API int fa_fwd_fp8_workspace_bytes(int B, int H_kv, int N, int d, unsigned long long* bytes);

/*
 * fa_fwd_host -- fa_fwd_ext on HOST buffers: the same operation (sources
 * as for fa_fwd_ext), with q, k, v read from host memory and o, lse written
 * back to host memory.
 *
 * The problem is cut into chunks of whole K/V-head groups (a K/V head with
 * the H / H_kv query heads that read it; about 8 chunks, each with at least
 * 4 MiB of input).  Each chunk is copied into a device staging slot, computed
 * by the forward kernel and copied back; up to three slots form a ring, so
 * that copying chunk i+1 in, computing chunk i and copying chunk i-1 out
 * overlap.  Copies run on two helper streams the library creates per device
 * on first use (kept for the life of the process), forked from `stream` and
 * joined back into it: the call is asynchronous, and all of its work,
 * copies included, is ordered after earlier work on `stream` and before
 * later work on it.  The result is bit-for-bit that of fa_fwd_ext on the
 * same inputs.
 *
 *   q, k, v, o, lse  host pointers with the layouts of fa_fwd_ext (lse may
 *            be NULL).  They should be page-locked (cudaHostAlloc or
 *            cudaHostRegister) for the copies to overlap; pageable memory
 *            works but each copy then runs synchronously with the host, and
 *            cannot be captured into a CUDA graph (FA_ERR_CUDA).  o and lse
 *            hold the result once `stream` has reached the end of the call's
 *            work; they must not overlap q, k or v.
 *   workspace, workspace_bytes
 *            device staging memory, 256-byte aligned (else
 *            FA_ERR_MISALIGNED); fa_fwd_host_workspace_bytes() gives the
 *            size of the default plan.  A smaller workspace is used with
 *            fewer groups per chunk, then fewer slots; FA_ERR_INVALID_ARG if
 *            one slot of one group does not fit.  Overwritten; need not be
 *            initialised; must not be used by other work until the call's
 *            work on `stream` is done.
 *   dtype    FA_DTYPE_F16 or FA_DTYPE_BF16.
 * Other arguments, validation and errors as in fa_fwd_ext; window bounds
 * below -1 are rejected (FA_ERR_INVALID_ARG).  Argument errors are reported
 * before anything is enqueued.  Concurrent calls on one device share the
 * helper streams (their enqueue is serialised by a lock).
 */
FA_API int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                       int window_right, int dtype, void* workspace,
                       unsigned long long workspace_bytes, void* stream);

/* Device staging bytes of fa_fwd_host's default plan for these sizes
 * (written to *bytes; with_lse 1 when lse is not NULL, else 0).  Empty
 * problems need 0 bytes. */
FA_API int fa_fwd_host_workspace_bytes(int B, int H, int H_kv, int N, int d, int with_lse,
                                       unsigned long long* bytes);

/*
 * fa_bwd -- attention backward pass: dQ, dK, dV from Q, K, V, the forward's
 * O and LSE, and dO.
 *
 * Source: flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp"
 * (CollectiveMainloopBwd::mma): P = exp(scale Q K^T - LSE), dP = dO V^T,
 * D = rowsum(dO * O) (the page's dPsum), dS = P (dP - D), dV = P^T dO,
 * dK = scale dS^T Q, dQ = scale dS K; grouped K/V heads sum their query
 * heads' dK and dV; masks and windows as in fa_fwd_ext.
 *
 *   q, o, dout, dq   contiguous [B][H][N][d] of `dtype` (o and lse as written
 *                    by fa_fwd_ext for the same arguments).
 *   k, v, dk, dv     contiguous [B][H_kv][N][d].
 *   lse              contiguous [B][H][N] float32 (natural log).
 *   workspace        device scratch of at least fa_bwd_workspace_bytes()
 *                    bytes, 256-byte aligned; overwritten, need not be
 *                    initialised.
 *   d                64 or 128 (else FA_ERR_UNSUPPORTED).
 * Every other argument, alignment rule and error is that of fa_fwd_ext (q,
 * k, v, o, dout, dq, dk, dv 16-byte aligned; lse 4-byte).  Enqueues three
 * kernels on `stream` (a row-sum pre-pass, the dK/dV kernel, the dQ kernel);
 * no atomics, so the gradients are bit-for-bit reproducible.  Allocates no
 * device memory.
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o,
                  const float* lse, const void* dout, void* dq, void* dk, void* dv,
                  void* workspace, unsigned long long workspace_bytes, int B, int H,
                  int H_kv, int N, int d, float scale, int causal, int window_left,
                  int window_right, int dtype, void* stream);

/*
 * fa_bwd_varlen -- fa_bwd over packed variable-length batches: q, o, dout, dq
 * are [total][H][d], k, v, dk, dv [total][H_kv][d], lse [H][total] (as written
 * by fa_fwd_varlen), with cu_seqlens, batch, max_seqlen and total as in
 * fa_fwd_varlen (offsets clamped by the kernels).  The workspace is
 * fa_bwd_workspace_bytes(batch, H, max_seqlen).  Rows outside every sequence
 * are not written.  Other rules as in fa_bwd.
 */
FA_API int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         const int* cu_seqlens, int batch, int max_seqlen, int total, int H,
                         int H_kv, int d, float scale, int causal, int window_left,
                         int window_right, int dtype, void* workspace,
                         unsigned long long workspace_bytes, void* stream);

/*
 * fa_bwd_varlen_qk -- the backward of fa_fwd_varlen_qk: separate query and key
 * sequences with optional used lengths (cross-attention, padded batches).
 *
 * Source: flash-attention "hopper/mainloop_bwd_sm90_tma_gmma_ws.hpp"
 * (CollectiveMainloopBwd::Arguments: cu_seqlens_q, cu_seqlens_k, seqused_q,
 * seqused_k; get_seqlen_q / get_seqlen_k; the causal and local masks shifted
 * by seqlen_k - seqlen_q).
 *
 *   q, o, dout, dq  [total_q][H][d]; lse [H][total_q] as written by
 *                   fa_fwd_varlen_qk (a row without keys has LSE = -inf).
 *   k, v, dk, dv    [total_k][H_kv][d].
 *   cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k, batch, max_seqlen_q,
 *   max_seqlen_k, total_q, total_k, causal, window_left, window_right
 *                   as in fa_fwd_varlen_qk (bottom-right aligned masks).
 *                   batch, max_seqlen_q or total_q 0: nothing is done.
 *   workspace       fa_bwd_workspace_bytes(batch, H, max_seqlen_q) bytes.
 *
 * Written: dQ for the used query rows of every sequence (0 for a row that
 * sees no key), dK and dV for the used key rows (0 for a key no query sees).
 * Rows past the used lengths and rows outside every sequence are not
 * written.  Passing one offset array for both (equal totals, no used
 * lengths) is fa_bwd_varlen.  Other rules as in fa_bwd.
 */
FA_API int fa_bwd_varlen_qk(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* seqused_q, const int* seqused_k, int batch,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                            int H, int H_kv, int d, float scale, int causal, int window_left,
                            int window_right, int dtype, void* workspace,
                            unsigned long long workspace_bytes, void* stream);

/* Workspace bytes of fa_bwd for these sizes (written to *bytes). */
FA_API int fa_bwd_workspace_bytes(int B, int H, int N, unsigned long long* bytes);

/* Human-readable name of a status code (static string, never NULL). */
FA_API const char* fa_status_string(int status);

/*
 * Synchronise `stream`, then read and clear the device status word that the
 * kernels' bounded waits set when one runs out.  Returns FA_OK,
 * FA_ERR_DEVICE_TIMEOUT, or FA_ERR_CUDA if the synchronisation failed; also
 * FA_ERR_MISALIGNED (site 13) if a backward kernel found its dynamic shared
 * memory not 1024-byte aligned and returned without doing anything.
 * `site` (may be NULL) receives the code of the wait that ran out (0 if none).
 */
FA_API int fa_get_device_status(void* stream, int* site);

/*
 * Set the limit of every device-side wait of later launches, in
 * microseconds (default 2,000,000 = 2 s; must be >= 1).  Not a compute
 * setting: only bounds how long a stalled pipeline stage waits before the
 * kernel gives up, records FA_ERR_DEVICE_TIMEOUT and returns.
 */
FA_API int fa_set_wait_timeout_us(long long timeout_us);

/*
 * Cap the persistent grid of later fa_fwd launches at `max_ctas` CTAs
 * (0 = one CTA per SM, the default).  Used by tests to run many work units
 * through each CTA on small inputs.
 */
FA_API int fa_set_max_ctas(int max_ctas);

/*
 * Watchdog self-test: launch one CTA that waits on an mbarrier nobody
 * arrives on, with a wait limit of `timeout_us`.  The kernel must give up,
 * record FA_ERR_DEVICE_TIMEOUT in the device status word and return; read it
 * with fa_get_device_status().  Faults nothing and traps nothing.
 */
FA_API int fa_selftest_watchdog(long long timeout_us, void* stream);

/*
 * Grouped-query packing of the packed-sequence forwards (fa_fwd_varlen,
 * fa_fwd_varlen_qk) at d <= 128: with enable = 1 (the default), when the
 * query heads share each K/V head in groups of 2, 4, 8 or 16, the g heads of
 * a group are packed into every 128-row tile (128 / g positions x g heads),
 * so that a group streams its keys and values once and short query
 * sequences (decoding) still fill the tiles; 0 computes each query head in
 * its own tiles.  The results agree within the parity tolerances (the
 * lazy rescale may pick a different reference maximum, so they are not bit
 * for bit the same).  A process-wide setting for later calls; FA_OK, or
 * FA_ERR_INVALID_ARG for another value.
 */
FA_API int fa_set_gqa_pack(int enable);

/* Number of SMs the persistent grid is sized from (current device), or -1. */
FA_API int fa_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
