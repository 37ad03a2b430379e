/*
 * fa.h — C ABI of exact, tiled attention for GB300 (sm_103a).
 *
 * The operation is exact attention, O = softmax(Q K^T * scale) V, with the
 * per-row log-sum-exp LSE kept for a backward pass ("FlashAttention: The
 * Matrix You Never Have to Write Down", section "What attention computes, in
 * one page" for the function, section "From softmax to attention: rescale
 * the output too" for the online recurrence the kernels run, section "Build
 * it" for the outputs O and L).  The N x N score or probability matrix is
 * never written to memory ("Why FlashAttention Can Avoid a Square Attention
 * Array Without Making Attention Linear", section "Tiles need a shared
 * softmax normalization").
 *
 * Entry points:
 *  - forward: fa_fwd (square), fa_fwd_ws / fa_fwd_static (the same, with the
 *    last round balanced through a caller's or the library's scratch),
 *    fa_fwd_kv (queries against a key set of another length, key counts,
 *    causal alignment, value width), fa_fwd_varlen (packed batches),
 *    fa_fwd_dropout, fa_fwd_kv_dropout, fa_fwd_varlen_dropout (dropout on
 *    the attention weights);
 *  - backward: fa_bwd, fa_bwd_kv, fa_bwd_varlen, fa_bwd_dropout,
 *    fa_bwd_kv_dropout, fa_bwd_varlen_dropout, each the gradient of the
 *    forward of the same name; fa_bwd_onepass, fa_bwd_onepass_dropout
 *    (fa_bwd and fa_bwd_dropout in one pass over the tiles, dQ summed
 *    through a caller's fp32 scratch);
 *  - decoding: fa_decode (a few queries against a long cache, key axis
 *    split across the GPU);
 *  - status and settings: fa_strerror, fa_status, fa_set_watchdog_ns,
 *    fa_set_unit_group, fa_watchdog_selftest, fa_work_tiles, fa_version.
 *
 * Conventions shared by every entry point (the kv, varlen and decode entry
 * points state their own layouts and alignments below):
 *  - Tensors are dense, contiguous, row-major, on the CURRENT CUDA device:
 *      q, k, v, o : [B, H, N, d] in the storage dtype (bf16 or fp16);
 *      lse        : [B, H, N] float32, natural log of the scaled scores.
 *  - The caller owns every buffer.  The library allocates no device memory
 *    and never builds an N x N buffer: workspaces (fa_fwd_ws, fa_decode)
 *    and the backward's per-row scratch are the caller's, O(SMs * 128 * d)
 *    or O(rows), never O(N^2); fa_fwd_static uses a fixed array of the
 *    library instead.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  A
 *    non-zero return means nothing was launched.
 *  - Causal masking of the square entry points is upper-left aligned: query
 *    i sees keys j <= i (section "Build it", note on non-square causal
 *    alignment); with equal query and key lengths this is also the
 *    bottom-right convention.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage dtype of q, k, v and o. */
typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/* Return codes.  They mirror the pages' raise-on-bad-input contract (section
 * "Build it", the input checks; section "Check it", the failing cases). */
enum {
  FA_OK = 0,
  FA_ERR_NULLPTR = 1,        /* a required pointer is NULL                     */
  FA_ERR_SHAPE = 2,          /* B, H or N negative, d <= 0, or sizes overflow  */
  FA_ERR_UNSUPPORTED_D = 3,  /* d is not 64 or 128                             */
  FA_ERR_DTYPE = 4,          /* dtype is not FA_BF16 / FA_FP16                 */
  FA_ERR_ALIGN = 5,          /* q/k/v/o not 16-byte aligned, lse not 4-byte    */
  FA_ERR_SCALE = 6,          /* scale not finite and > 0                       */
  FA_ERR_DEVICE = 7,         /* current device is not a compute 10.3 GPU       */
  FA_ERR_TENSORMAP = 8,      /* the driver refused a TMA descriptor            */
  FA_ERR_LAUNCH = 9,         /* the launch itself failed (CUDA error)          */
  FA_ERR_TIMEOUT = 10,       /* a kernel's bounded wait ran out (fa_status)    */
  FA_ERR_CUDA = 11,          /* a CUDA runtime call failed (fa_status)         */
  FA_ERR_WORKSPACE = 12,     /* workspace smaller than fa_fwd_workspace_size   */
  FA_ERR_DROPOUT = 13        /* dropout probability outside [0, 1 - 1/512)     */
};

/*
 * fa_fwd — exact attention forward.
 *
 * Computes the function of "FlashAttention: The Matrix You Never Have to
 * Write Down", section "What attention computes, in one page" (scores
 * scale * q_i . k_j, a softmax over each row, the weighted sum of the
 * values), by the online recurrence of section "From softmax to attention:
 * rescale the output too" over 128 x 128 tiles, and returns the two outputs
 * of section "Build it": O, and the per-row log-sum-exp L kept for the
 * backward pass.  Causal calls skip key tiles wholly in a query tile's
 * future and mask only the diagonal tile (section "Causal masking: half the
 * score tiles disappear").
 *
 *   q, k, v : device pointers, [B, H, N, d], dtype `dtype`, 16-byte aligned.
 *   o       : device pointer, [B, H, N, d], dtype `dtype`, 16-byte aligned;
 *             O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) v_j, rounded to
 *             nearest-even in the storage dtype.
 *   lse     : device pointer, [B, H, N] float32, 4-byte aligned;
 *             LSE[b,h,i] = ln sum_j exp(scale * q_i . k_j).
 *   B, H, N : batch, heads, sequence length (queries = keys = N).  Any N >= 0;
 *             a ragged last tile is masked.  B*H*N == 0 writes nothing and
 *             returns FA_OK without touching the pointers.
 *   d       : head width, 64 or 128.
 *   causal  : nonzero for the causal mask (key j visible to query i iff j <= i).
 *   scale   : multiplier of q.k, finite and > 0 (usually 1/sqrt(d)).
 *   dtype   : FA_BF16 or FA_FP16 (q, k, v, o share it).
 *   stream  : CUDA stream the kernel is enqueued on.
 *
 * Errors: FA_ERR_SHAPE, FA_ERR_UNSUPPORTED_D, FA_ERR_DTYPE, FA_ERR_SCALE are
 * checked first, then the empty case, then FA_ERR_NULLPTR, FA_ERR_ALIGN,
 * FA_ERR_DEVICE, FA_ERR_TENSORMAP, FA_ERR_LAUNCH.  Errors that happen on the
 * device after the launch are reported by fa_status().
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int N, int d, int causal, float scale, int dtype,
           cudaStream_t stream);

/*
 * fa_fwd_kv — exact attention of Nq queries against a key set of its own
 * length, with per-batch key counts (padding) and an explicit causal
 * alignment.
 *
 * The pages' square formulation puts query i at absolute position i
 * (upper-left alignment) and name two extensions it leaves out: non-square
 * causal alignment with query positions offset by the cache length (for
 * incremental decoding and chunked prefill), and masks such as padding
 * under which a query row can see no key at all, which then needs a stated
 * policy ("FlashAttention: The Matrix You Never Have to Write Down",
 * section "Two things this deliberately doesn't do"; the empty key set's
 * policy, O = 0 and LSE = -inf, in the same page's reference
 * implementation).  This entry point does both with the same tiled online
 * softmax as fa_fwd.  It also takes a value width dv different from the
 * query/key width d: the same page's reference lets V be wider or narrower
 * than Q and K and tests shapes with dv != d (section "Check it", the sweep
 * over shapes and block sizes).
 *
 *   q         : device pointer, [B, H, Nq, d], dtype `dtype`, 16-byte aligned.
 *   k         : device pointer, [B, H, Nk, d], 16-byte aligned.
 *   v         : device pointer, [B, H, Nk, dv], 16-byte aligned (k and v may
 *               be NULL when Nk = 0).
 *   o         : device pointer, [B, H, Nq, dv], 16-byte aligned (written).
 *   lse       : device pointer, [B, H, Nq] float32, 4-byte aligned (written).
 *   Nq, Nk    : queries and key capacity per head (>= 0).
 *   d, dv     : widths of Q/K and of V/O, each 64 or 128.  With d != dv the
 *               kernel of width 128 runs; it loads only each tensor's own
 *               columns, S takes only d's products and O += P V computes
 *               only dv's columns.
 *   seqlens_k : NULL (every batch has Nk keys) or a device pointer to B
 *               int32 key counts, 4-byte aligned; batch b uses keys
 *               0 .. len_b - 1 (values are clamped to [0, Nk]); the rest
 *               is padding and never contributes.
 *   causal    : 0 no mask; 1 upper-left (query i at position i); 2
 *               bottom-right (query i at position len_b - Nq + i: the
 *               queries are the last Nq positions of the batch's keys).
 *               Key j is visible to a query at position q_pos iff j <= q_pos.
 *   A query row that sees no key gets O = 0 and LSE = -inf.
 *   scale, dtype, stream : as fa_fwd.
 *
 * Errors as fa_fwd (FA_ERR_UNSUPPORTED_D for d or dv outside {64, 128});
 * FA_ERR_SHAPE also when causal is not 0, 1 or 2; FA_ERR_ALIGN also for a
 * misaligned seqlens_k.  B*H*Nq == 0 writes nothing.
 */
int fa_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int H, int Nq, int Nk, int d, int dv, int causal,
              const int *seqlens_k, float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_varlen — exact attention over a packed batch of sequences of
 * different lengths, with no padding.
 *
 * The pages point out that padding every sequence of a batch to the longest
 * one makes a fused kernel do work for the padded positions, and that at
 * mixed lengths packing or a variable-length kernel matters more than the
 * choice of attention implementation ("FlashAttention: The Matrix You Never
 * Have to Write Down", section on PyTorch's scaled_dot_product_attention,
 * the padding note).  This entry point runs the same tiled online softmax
 * as fa_fwd_kv on packed tensors: each sequence attends only to its own
 * keys, and no tile is spent past a sequence's end.
 *
 *   q            : device pointer, [total_q, H, d], dtype `dtype`, 16-byte aligned.
 *   k            : device pointer, [total_k, H, d], 16-byte aligned.
 *   v            : device pointer, [total_k, H, dv], 16-byte aligned (k and v
 *                  may be NULL when total_k = 0).
 *   o            : device pointer, [total_q, H, dv], 16-byte aligned (written).
 *   lse          : device pointer, [H, total_q] float32, 4-byte aligned (written).
 *   cu_seqlens_q : device pointer, B + 1 int32, 4-byte aligned: sequence b
 *                  owns query tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1] - 1.
 *   cu_seqlens_k : the same for key/value tokens.
 *                  Offsets are clamped to [0, total] and an end below its
 *                  start counts as an empty sequence, so no value of these
 *                  arrays makes the kernel read or write out of bounds;
 *                  overlapping sequences are the caller's error.
 *   max_seqlen_q : an upper bound on every sequence's query count (sizes the
 *                  grid); query rows past it are not computed.
 *   total_q, total_k : packed token counts (>= 0).
 *   d, dv        : widths of Q/K and of V/O, each 64 or 128.
 *   causal       : 0 none; 1 upper-left (query i of a sequence at position
 *                  i); 2 bottom-right (at position len_k - len_q + i), per
 *                  sequence.  A query row that sees no key gets O = 0 and
 *                  LSE = -inf.
 *   scale, dtype, stream : as fa_fwd.
 *
 * Errors as fa_fwd_kv; FA_ERR_NULLPTR also for missing cu_seqlens arrays,
 * FA_ERR_ALIGN also for misaligned ones.  B*H == 0, max_seqlen_q == 0 or
 * total_q == 0 writes nothing.
 */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int total_q, int total_k, int d, int dv, int causal,
                  float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_dropout — fa_fwd with dropout on the attention weights, the mask
 * drawn from a counter-based generator whose state (seed, offset) is all
 * the backward pass needs to draw it again.
 *
 * The pages: with dropout enabled, the full algorithm keeps the
 * pseudorandom generator's state so that backward regenerates the same
 * dropout mask instead of storing a square mask ("Why FlashAttention Can
 * Avoid a Square Attention Array Without Making Attention Linear", section
 * "Backward can recreate tiles instead of retaining the square").  The
 * generator and the keep rule are this library's reading:
 *   - Philox4x32-10 (Salmon et al., SC 2011); one call per 4 x 4 block of a
 *     head's attention matrix, counter (key / 4, query / 4, b * H + h,
 *     offset), key = seed (low word first); element (i, j) takes byte j % 4
 *     of output word i % 4;
 *   - kept when that byte < t = floor((1 - dropout_p) * 256 + 1/2) (keep
 *     probability t / 256), kept weights scaled by 256 / t;
 *   - the softmax normalisation and LSE are those without dropout:
 *     O_i = (256 / t) sum_j exp(s_ij - m_i) Z_ij V_j / l_i.
 *
 *   dropout_p : in [0, 1) with t >= 1; 0 runs fa_fwd (bit-identical).
 *   seed, offset : generator state; the same values in fa_bwd_dropout
 *               give the same mask.  Use a new offset (or seed) per call
 *               that should draw a new mask.
 *   causal    : 0 or 1 (upper-left; the shapes are square).
 *   Other arguments, layouts and errors as fa_fwd; FA_ERR_DROPOUT for a
 *   dropout_p outside the range.
 */
int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int N, int d, int causal, float scale, float dropout_p,
                   unsigned long long seed, unsigned int offset, int dtype,
                   cudaStream_t stream);

/*
 * fa_fwd_ws — fa_fwd with a caller-provided workspace used to balance the
 * last round of work across all SMs.
 *
 * The persistent kernel deals whole (batch*head, 256-row query block) units
 * to the SMs; when the units do not fill whole rounds, the last units are
 * cut along the key axis so every SM does the same number of key tiles, and
 * the partial results of a cut unit (unnormalised O, running max m and sum
 * l per row, kept in the workspace) are combined by the identity the online
 * softmax rests on: rescale every part to the largest m, add, divide once
 * ("FlashAttention: The Matrix You Never Have to Write Down", section "What
 * it doesn't solve", on splitting the key axis across workers and combining
 * partial results).  Results equal fa_fwd's up to rounding order.
 *
 *   workspace, workspace_bytes : device buffer, 256-byte aligned, at least
 *       the size fa_fwd_workspace_size reports for the same shape on the
 *       current device.  Owned by the caller; its contents need no
 *       initialisation and are not meaningful after the call.  Calls that
 *       share one workspace must not overlap on the GPU (use one workspace
 *       per stream).  NULL (or a shape that needs none) runs fa_fwd.
 *   Other arguments, errors and asynchrony as fa_fwd; FA_ERR_WORKSPACE when
 *   the workspace is too small, FA_ERR_ALIGN when it is misaligned.
 * Causal calls, and calls whose units fill whole rounds, use no workspace.
 */
int fa_fwd_ws(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int H, int N, int d, int causal, float scale, int dtype,
              void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_workspace_size — bytes of workspace fa_fwd_ws needs for this shape
 * on the current device (0 when it would not split anything).  Returns
 * FA_ERR_NULLPTR, FA_ERR_SHAPE, FA_ERR_UNSUPPORTED_D or FA_ERR_DEVICE.
 */
int fa_fwd_workspace_size(int B, int H, int N, int d, int causal, size_t *bytes);

/*
 * fa_fwd_static — fa_fwd_ws for callers that cannot allocate device memory.
 *
 * The pages have no counterpart; this is an integration convenience.  Some
 * callers only ever see raw device pointers and have no allocator of their
 * own to get a workspace from (a plugin or launch hook inside a host
 * framework that owns all device memory), and some must not call cudaMalloc
 * on their path at all (it can synchronise the whole device, which a
 * latency-bound loop cannot afford).  This entry point allocates nothing: it
 * runs fa_fwd_ws with a 40 MiB scratch array that the library keeps on every
 * GPU it is loaded on, from load until the process exits.
 *
 *   Arguments, results and errors as fa_fwd_ws, without the workspace, and
 *   checked in the same order; FA_ERR_WORKSPACE (after those checks) when
 *   the shape needs more than the 40 MiB array holds (no supported shape
 *   does on a GPU with up to 152 SMs).
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   A device reset (cudaDeviceReset) replaces the device's context and
 *   reloads the library's code there; the next call notices the new context
 *   and looks the address up again, so that call too belongs outside any
 *   capture.
 *   Every call on a device shares the one array and leaves its last contents
 *   in it (the counters that must start at zero are cleared by each call):
 *   calls that overlap on the GPU — other streams, other host threads —
 *   race on it and must be serialised by the caller.
 */
int fa_fwd_static(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int N, int d, int causal, float scale, int dtype,
                  cudaStream_t stream);

/*
 * fa_bwd — gradients of exact attention: dQ, dK, dV of sum(dO * O) for the
 * O that fa_fwd computes from the same q, k, v, causal and scale.
 *
 * The pages describe the backward pass as keeping Q, K, V, the output O and
 * the per-row statistics L, and rebuilding the score and probability tiles
 * from them rather than storing the N x N matrices ("FlashAttention: The
 * Matrix You Never Have to Write Down", section "The forward pass is only
 * half of it"; "Why FlashAttention Can Avoid a Square Attention Array
 * Without Making Attention Linear", section "Backward can recreate tiles
 * instead of retaining the square").  With P = exp(scale q.k - LSE) and
 * D = rowsum(dO * O): dV = P^T dO, dS = P * (dO V^T - D), dQ = scale dS K,
 * dK = scale dS^T Q.  No N x N buffer is allocated or written.
 *
 *   q, k, v, o : device pointers, [B, H, N, d], dtype `dtype`, 16-byte
 *                aligned; o is the fa_fwd output for q, k, v.
 *   lse        : device pointer, [B, H, N] float32, the fa_fwd LSE.
 *   dout       : device pointer, [B, H, N, d], dtype `dtype`: dLoss/dO.
 *   dq, dk, dv : device pointers, [B, H, N, d], dtype `dtype`, 16-byte
 *                aligned, written (rounded to nearest-even).
 *   delta      : device pointer, [B, H, N] float32, 4-byte aligned, owned
 *                by the caller: written with D = rowsum(dO * O) and read
 *                back by the gradient kernels (scratch for the caller).
 *   B, H, N, d, causal, scale, dtype, stream : as fa_fwd.
 * Errors and asynchrony as fa_fwd (FA_ERR_NULLPTR for any of the ten
 * pointers).  Results are deterministic: every gradient row is written by
 * one CTA, without atomics.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, float *delta,
           int B, int H, int N, int d, int causal, float scale, int dtype,
           cudaStream_t stream);

/*
 * fa_bwd_onepass — the gradients fa_bwd computes, with every (query tile,
 * key tile) pair visited once.  The same passages define them (tiles are
 * rebuilt from Q, K, V, O and the row statistics, never stored: "Why
 * FlashAttention Can Avoid a Square Attention Array Without Making
 * Attention Linear", section "Backward can recreate tiles instead of
 * retaining the square").  fa_bwd forms S and dP twice, once for dK/dV
 * (per key tile) and once for dQ (per query tile).  Here the per-key-tile
 * pass also forms dQ_i = dS K_j and adds it in fp32 into the caller's
 * scratch; a final kernel writes dQ = scale * sum.  That is five tile
 * products per pair instead of seven.  The fp32 additions of different key
 * tiles land in an unspecified order, so dQ can differ from call to call in
 * its last bits (dK and dV cannot: each of their rows has one writer).
 *
 *   q ... dtype, stream : as fa_bwd (d 64 or 128).
 *   workspace       : device pointer, 16-byte aligned, at least
 *                     fa_bwd_onepass_workspace_size bytes, owned by the
 *                     caller; zeroed and overwritten on `stream` by every
 *                     call.  Must not be in use by other work meanwhile.
 *   workspace_bytes : its size in bytes.
 * Errors as fa_bwd, plus FA_ERR_WORKSPACE for a missing or short workspace
 * and FA_ERR_ALIGN for a misaligned one (checked after the arguments
 * fa_bwd checks; nothing is launched then).
 */
int fa_bwd_onepass(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dout, void *dq, void *dk, void *dv,
                   float *delta, int B, int H, int N, int d, int causal, float scale,
                   int dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_onepass_dropout — fa_bwd_dropout computed as fa_bwd_onepass does:
 * each (query tile, key tile) pair is visited once and the forward's mask is
 * drawn once for it from the same dropout_p, seed and offset.  dK and dV
 * equal fa_bwd_dropout's bit for bit; dQ is summed in fp32 through
 * `workspace` in no fixed order.  Arguments as fa_bwd_dropout plus workspace
 * and workspace_bytes (as fa_bwd_onepass); errors as fa_bwd_onepass plus
 * FA_ERR_DROPOUT (checked first) for a dropout_p outside [0, 1) or leaving
 * t = 0.
 */
int fa_bwd_onepass_dropout(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dout, void *dq, void *dk, void *dv,
                           float *delta, int B, int H, int N, int d, int causal, float scale,
                           float dropout_p, unsigned long long seed, unsigned int offset,
                           int dtype, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * fa_bwd_onepass_workspace_size — bytes of the fp32 dQ sum of
 * fa_bwd_onepass and fa_bwd_onepass_dropout: B * H * d * (N rounded up to a
 * multiple of 128) * 4.
 * Host-only.  Returns FA_ERR_NULLPTR for a NULL `bytes`, FA_ERR_SHAPE for a
 * negative B, H or N, FA_ERR_UNSUPPORTED_D for d other than 64 or 128.
 */
int fa_bwd_onepass_workspace_size(int B, int H, int N, int d, size_t *bytes);

/*
 * fa_bwd_kv — the backward pass of fa_fwd_kv: dQ, dK, dV of sum(dO * O) for
 * O, LSE = fa_fwd_kv(q, k, v, ...) with the same Nq, Nk, widths, key counts
 * and causal alignment.  The pages give the backward's
 * principle (keep Q, K, V, O and the row statistics, rebuild the tiles;
 * "Why FlashAttention Can Avoid a Square Attention Array Without Making
 * Attention Linear", section "Backward can recreate tiles instead of
 * retaining the square"); the masks are fa_fwd_kv's.
 *
 *   q, dq          : [B, H, Nq, d];  k, dk : [B, H, Nk, d];
 *   o, dout        : [B, H, Nq, dv_width];  v, dv : [B, H, Nk, dv_width];
 *   d, dv_width    : 64 or 128 each (the value width may differ from the
 *                    query/key width, as in fa_fwd_kv; first page, section
 *                    "Check it", shapes with dv != d);
 *   lse, delta     : [B, H, Nq] float32 (delta is scratch, as in fa_bwd).
 *   seqlens_k, causal (0, 1 upper-left, 2 bottom-right) : as fa_fwd_kv.
 *   Keys that no query sees (padding past a batch's key count, or keys
 *   after every query's position) get dK = dV = 0; query rows that see no
 *   key get dQ = 0.  k, v, dk, dv may be NULL when Nk = 0, and q, o, dout,
 *   dq, lse, delta when Nq = 0.
 *   Errors as fa_bwd; FA_ERR_SHAPE also for causal outside 0 .. 2.
 */
int fa_bwd_kv(const void *q, const void *k, const void *v, const void *o, const float *lse,
              const void *dout, void *dq, void *dk, void *dv, float *delta,
              int B, int H, int Nq, int Nk, int d, int dv_width, int causal,
              const int *seqlens_k, float scale, int dtype, cudaStream_t stream);

/*
 * fa_bwd_varlen — the backward pass of fa_fwd_varlen (packed batches of
 * sequences of different lengths): dQ, dK, dV of sum(dO * O) for O, LSE =
 * fa_fwd_varlen(...) with the same offsets, widths and causal mode; each
 * sequence's gradients come from its own queries and keys only.
 *
 *   q, dq : [total_q, H, d];  k, dk : [total_k, H, d];
 *   o, dout : [total_q, H, dv_width];  v, dv : [total_k, H, dv_width]
 *   (d and dv_width 64 or 128 each).
 *   lse            : [H, total_q] float32, as fa_fwd_varlen wrote it.
 *   delta          : [total_q, H] float32 scratch (written, as in fa_bwd).
 *   cu_seqlens_q, cu_seqlens_k : the forward's offset arrays (clamped the
 *                  same way, so no value of them reads or writes out of
 *                  bounds).
 *   max_seqlen_q, max_seqlen_k : upper bounds on every sequence's query and
 *                  key counts (they size the grid).
 *   Keys no query sees get dK = dV = 0, query rows that see no key dQ = 0.
 *   Errors as fa_fwd_varlen.
 */
int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, float *delta,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int d,
                  int dv_width, int causal, float scale, int dtype, cudaStream_t stream);

/*
 * fa_bwd_dropout — fa_bwd for an output of fa_fwd_dropout: the same
 * dropout_p, seed and offset regenerate the forward's mask on the device
 * (nothing square is stored or read), and with Z the keep mask and
 * s = 256 / t:  dV_j = s sum_i P_ij Z_ij dO_i,  dP_ij = s Z_ij dO_i . V_j,
 * dS = P (dP - D) with D = rowsum(dO * O) as in fa_bwd.
 * Arguments, layouts and errors as fa_bwd; FA_ERR_DROPOUT for a dropout_p
 * outside [0, 1) or leaving t = 0.
 */
int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                   const float *lse, const void *dout, void *dq, void *dk, void *dv,
                   float *delta, int B, int H, int N, int d, int causal, float scale,
                   float dropout_p, unsigned long long seed, unsigned int offset, int dtype,
                   cudaStream_t stream);

/*
 * fa_fwd_kv_dropout, fa_fwd_varlen_dropout — fa_fwd_kv and fa_fwd_varlen with
 * dropout on the attention weights, the mask drawn on the device from
 * (seed, offset) as in fa_fwd_dropout ("Why FlashAttention Can Avoid a
 * Square Attention Array Without Making Attention Linear", section
 * "Backward can recreate tiles instead of retaining the square": the
 * generator's state is kept so the backward pass regenerates the mask).
 * Element (i, j) of a (batch, head) — with packed batches a (sequence,
 * head) — is drawn by its query row i and key index j within that pair,
 * whatever the causal alignment: the alignment only decides which keys a
 * row sees.  dropout_p = 0 gives fa_fwd_kv's (fa_fwd_varlen's) result.
 * Arguments and errors as those entry points plus dropout_p, seed, offset
 * and FA_ERR_DROPOUT as in fa_fwd_dropout.
 *
 * fa_bwd_kv_dropout, fa_bwd_varlen_dropout — the matching backward passes
 * (the same dropout_p, seed and offset as the forward call): arguments and
 * errors as fa_bwd_kv and fa_bwd_varlen plus those three.
 */
int fa_fwd_kv_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int H, int Nq, int Nk, int d, int dv, int causal,
                      const int *seqlens_k, float scale, float dropout_p,
                      unsigned long long seed, unsigned int offset, int dtype,
                      cudaStream_t stream);
int fa_fwd_varlen_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                          const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                          int max_seqlen_q, int total_q, int total_k, int d, int dv,
                          int causal, float scale, float dropout_p, unsigned long long seed,
                          unsigned int offset, int dtype, cudaStream_t stream);
int fa_bwd_kv_dropout(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv,
                      float *delta, int B, int H, int Nq, int Nk, int d, int dv_width,
                      int causal, const int *seqlens_k, float scale, float dropout_p,
                      unsigned long long seed, unsigned int offset, int dtype,
                      cudaStream_t stream);
int fa_bwd_varlen_dropout(const void *q, const void *k, const void *v, const void *o,
                          const float *lse, const void *dout, void *dq, void *dk, void *dv,
                          float *delta, const int *cu_seqlens_q, const int *cu_seqlens_k,
                          int B, int H, int max_seqlen_q, int max_seqlen_k, int total_q,
                          int total_k, int d, int dv_width, int causal, float scale,
                          float dropout_p, unsigned long long seed, unsigned int offset,
                          int dtype, cudaStream_t stream);

/*
 * fa_decode — attention of a few new queries against a long key/value cache
 * (decoding), with the key axis split across the GPU.
 *
 * With one (or a few) queries against N cached keys there is no square
 * score matrix to avoid; the call is bound by reading K and V and by finding
 * parallelism, so the key axis is split across many CTAs, each keeping the
 * online-softmax state (m, l, unnormalised O) of its key range, and the
 * parts are combined with the rescale identity: each part scaled to the
 * largest m, summed, divided once ("FlashAttention: The Matrix You Never
 * Have to Write Down", section "What it doesn't solve", on decoding and on
 * Flash-Decoding splitting the key axis and combining partial results).
 *
 *   q        : device pointer, [B, H, Nq, d], 1 <= Nq <= 16, 16-byte aligned.
 *   k, v     : device pointers, [B, H, Nk, d], the cache, 16-byte aligned
 *              (may be NULL when Nk == 0).
 *   o        : device pointer, [B, H, Nq, d], written in the storage dtype.
 *   lse      : device pointer, [B, H, Nq] float32, natural-log LSE.
 *   causal   : nonzero: query i sits at position Nk - Nq + i, after the
 *              cached keys, and sees keys j <= that position (the decoding
 *              convention: query positions offset by the cache length;
 *              section "Build it", note on non-square causal alignment).
 *   workspace, workspace_bytes : device buffer, 256-byte aligned, at least
 *              fa_decode_workspace_size bytes (partial results), owned by
 *              the caller; contents need no initialisation.  Calls sharing
 *              one workspace must not overlap on the GPU.
 *   scale, dtype, stream : as fa_fwd.
 * Nk == 0 writes O = 0 and LSE = -inf (the pages' empty-key policy), and so
 * does a causal query whose position is negative (Nq > Nk).
 * Errors: FA_ERR_SHAPE (also for Nq outside 1..16), FA_ERR_UNSUPPORTED_D,
 * FA_ERR_DTYPE, FA_ERR_SCALE, then B*H == 0 returns FA_OK, then
 * FA_ERR_NULLPTR, FA_ERR_ALIGN, FA_ERR_DEVICE, FA_ERR_WORKSPACE,
 * FA_ERR_TENSORMAP, FA_ERR_LAUNCH.
 */
int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int H, int Nq, int Nk, int d, int causal, float scale, int dtype,
              void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_decode_workspace_size — bytes of workspace fa_decode needs for this
 * shape on the current device (0 when Nk == 0 or B*H == 0).  Returns
 * FA_ERR_NULLPTR, FA_ERR_SHAPE, FA_ERR_UNSUPPORTED_D or FA_ERR_DEVICE.
 */
int fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, size_t *bytes);

/*
 * fa_strerror — human-readable name of a return code (a static string, never
 * NULL; "unknown error code" for a value outside the enum).  The codes are
 * the C form of the input contract of "FlashAttention: The Matrix You Never
 * Have to Write Down": section "Build it" (its validation function raises on
 * a bad rank, width, length or dtype before any work) and section "Check
 * it" (the failing cases it expects to raise).  Codes from FA_ERR_DEVICE on
 * concern the GPU and have no counterpart there.
 */
const char *fa_strerror(int code);

/*
 * fa_status — device-side error state of kernels launched so far.
 *
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Every wait inside the kernels is bounded by a
 * watchdog; when one runs out the kernel records it there, finishes without
 * hanging (its outputs are then undefined) and this call returns
 * FA_ERR_TIMEOUT.  Returns FA_OK when no kernel reported a problem, FA_ERR_CUDA
 * if the synchronisation or the read failed.  `detail` (may be NULL) receives
 * the raw status word (bit 0: timeout; bits 8..15: id of the first wait that
 * ran out).
 */
int fa_status(cudaStream_t stream, unsigned int *detail);

/*
 * fa_set_watchdog_ns — budget of every bounded wait in kernels launched after
 * this call, in nanoseconds (default 2e9 = 2 s).  0 restores the default.
 * Host-side setting shared by all threads of the process.
 */
void fa_set_watchdog_ns(unsigned long long ns);

/*
 * fa_set_unit_group — override of the forward kernels' unit order (the pages
 * have no counterpart; it changes only which CTA computes which block, never
 * a result).  The persistent forward kernels deal (batch*head, 256-row query
 * block) units to the SMs from groups of `heads` heads, level by level inside
 * a group (the heaviest query block of each head of the group first).  0
 * (the default) lets each call choose: the largest group whose K/V fit an L2
 * budget, and for causal calls of known lengths the group whose simulated
 * deal is most even.  A positive value is used as is (clamped to B*H) by
 * every fa_fwd, fa_fwd_ws, fa_fwd_static, fa_fwd_kv and fa_fwd_varlen
 * launched afterwards.  Host-side setting shared by all threads of the
 * process.  Returns FA_ERR_SHAPE for a negative value.
 */
int fa_set_unit_group(int heads);

/*
 * fa_watchdog_selftest — failure-detection self-test (the pages have no
 * counterpart).  Launches on `stream` a one-thread kernel whose bounded
 * wait, the same routine every kernel of this library waits with, is on a
 * barrier that nothing ever completes.  The wait runs out after
 * `budget_ns` nanoseconds (1 .. 1e9) and records a timeout with site 31 in
 * the status word; fa_status then returns FA_ERR_TIMEOUT.  No fault, trap
 * or hang is involved, and the context stays usable.
 * Returns FA_ERR_SHAPE for a budget outside 1 .. 1e9, FA_ERR_DEVICE, or
 * FA_ERR_LAUNCH.
 */
int fa_watchdog_selftest(unsigned long long budget_ns, cudaStream_t stream);

/*
 * fa_work_tiles — host-side count of the (query tile, key tile) pairs the
 * forward kernel computes for one head with 128-row tiles, obtained by
 * walking that head's units through the kernel's own unit decoder (the same
 * function the kernel uses for its loop bounds): n^2 unmasked, or n(n+1)/2
 * causal with n = ceil(N/128) (section "Causal masking: half the score tiles
 * disappear": whole future tiles are skipped, diagonal tiles are masked).
 * Writes the count to *pairs.  Returns FA_ERR_SHAPE for N < 0,
 * FA_ERR_NULLPTR for a NULL `pairs`.
 */
int fa_work_tiles(int N, int causal, long long *pairs);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
