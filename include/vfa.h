/*
 * vfa.h -- C ABI of libvfa: variable-length FlashAttention forward and paged
 * GQA decode for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument named as a device buffer is a CUDA device
 *     address on the current device, allocated and owned by the caller.  The
 *     library never allocates, frees or retains caller memory, and keeps no
 *     pointer after a call returns.
 *   - Calls are asynchronous: they enqueue work on `stream` (NULL means the
 *     legacy default stream) and return.  Results are ready when the stream
 *     has reached that point.
 *   - Host-detected errors (null or misaligned pointers, unsupported sizes,
 *     a too-small workspace, a device that is not compute capability 10.3)
 *     return a non-zero vfa_status immediately and enqueue nothing.
 *     vfa_last_error() then describes the problem.
 *   - Data errors that only the device can see (cu_seqlens that are not a
 *     valid prefix sum, a block id outside the pool, a tile count above the
 *     tile capacity) never fault or trap: the kernels record a status code
 *     in a device status word, skip the offending work and leave its outputs
 *     untouched.  vfa_read_status() fetches that word.
 *   - bf16 means IEEE bfloat16 (1-8-7); f32 is IEEE binary32.
 */
#ifndef VFA_H
#define VFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *vfa_stream_t;

typedef enum {
    VFA_OK = 0,
    VFA_ERR_INVALID_ARG = 1,   /* host: null/misaligned pointer, bad size        */
    VFA_ERR_UNSUPPORTED = 2,   /* host: a size this build does not implement     */
    VFA_ERR_ARCH = 3,          /* host: the current device is not sm_103         */
    VFA_ERR_CUDA = 4,          /* host: a CUDA runtime call failed               */
    VFA_ERR_BAD_SEQLENS = 5,   /* device: cu_seqlens not a valid prefix sum      */
    VFA_ERR_BAD_BLOCK = 6,     /* device: block id or tile count out of range    */
    VFA_ERR_TIMEOUT = 7,       /* device: a bounded wait inside a kernel expired */
    VFA_ERR_WORKSPACE = 8      /* device: the work list does not fit the workspace */
} vfa_status;

/* Message for the last non-OK status returned on the calling host thread. */
const char *vfa_last_error(void);

/* Library version string, e.g. "vfa 0.1 sm_103a". */
const char *vfa_version(void);

/* ------------------------------------------------------------------------ */
/* Variable-length attention forward                                         */
/* ------------------------------------------------------------------------ */

/*
 * Workspace bytes vfa_varlen_fwd needs for these sizes (an upper bound that
 * holds for any cu_seqlens with these totals).  The first int32 of the
 * workspace is the call's device status word (see vfa_read_status).
 */
size_t vfa_varlen_fwd_workspace_bytes(int batch, int total_q, int total_k, int num_heads,
                                      int head_dim);

/*
 * Tile shape the forward uses for `head_dim`: q tile rows (*block_q), key
 * tile rows (*block_k), and whether one work item holds two q tiles
 * (*pair_tiles, 0 or 1).  The work list is built over these tiles.
 * Returns VFA_ERR_UNSUPPORTED for a head_dim this build does not implement.
 */
vfa_status vfa_varlen_fwd_tile_shape(int head_dim, int *block_q, int *block_k, int *pair_tiles);

/*
 * Exact softmax(scale * Q K^T, optional causal mask) V over packed
 * variable-length sequences, plus the per-(token, head) log-sum-exp.
 *
 * Defined by "Varlen Flash Attention Implementation Plan" (rustytorch),
 * Task 1 Step 1 (kernel preconditions, packed layout, masks, online-softmax
 * recurrence and the out / lse epilogue) and Task 2 Step 1 (the CPU
 * reference it must agree with).  The plan's kernel takes one block per
 * (global q tile, head); this library instead builds a per-sequence q-tile
 * work list on the device and covers every query row.
 *
 * q            device bf16 [total_q, num_heads, head_dim], packed row-major.
 * k, v         device bf16 [total_k, num_kv_heads, head_dim]; query head h
 *              reads kv head h / (num_heads / num_kv_heads) (grouped-query
 *              attention; num_kv_heads == num_heads is the plan's layout).
 * cu_seqlens_q device int32 [batch + 1]: 0, running sums of the q lengths;
 *              cu_seqlens_q[batch] == total_q.  Sequence b owns q rows
 *              [cu_seqlens_q[b], cu_seqlens_q[b+1]).
 * cu_seqlens_k device int32 [batch + 1], the same for keys/values.
 * total_q, total_k  the tensors' first extents (needed on the host to describe
 *              the tensors to the TMA engine).
 * max_seqlen_q an upper bound on every q length (checked on the device).
 * softmax_scale the factor applied to q.k before the softmax.
 * causal       0: no mask; 1: top-left causal mask in local positions --
 *              local key j is visible to local query i iff j <= i (the
 *              plan's kernel); 2: bottom-right -- j <= i + Lk_b - Lq_b, so the
 *              last query sees every key (a query block at the end of a longer
 *              key sequence) and rows with i + Lk_b - Lq_b < 0 see none.
 *              Other values: VFA_ERR_INVALID_ARG.
 * window_left  < 0: no window.  >= 0 (needs causal 1 or 2, else
 *              VFA_ERR_INVALID_ARG): a sliding window -- local key j is
 *              visible to local query i only if j >= i + off - window_left
 *              as well (off = 0 top-left, Lk_b - Lq_b bottom-right), so each
 *              query sees at most window_left + 1 keys ending at its
 *              diagonal.  The pages name sliding-window masks among the
 *              varlen variants without defining one; this is the reading
 *              taken.
 * out          device bf16 [total_q, num_heads, head_dim]: out = sum_j p_j v_j /
 *              sum_j p_j, rounded to nearest even; 0 for a query with no
 *              visible key.
 * lse          device f32 [total_q, num_heads]: natural-log sum of
 *              exp(scale * q.k_j) over visible keys; -FLT_MAX when there is
 *              none.
 * workspace    device scratch of at least vfa_varlen_fwd_workspace_bytes()
 *              bytes, 256-byte aligned; reused across calls; calls that share
 *              one workspace must be stream-ordered.
 *
 * Supported: head_dim in {64, 128, 256}; num_heads >= 1, a multiple of
 * num_kv_heads >= 1; batch >= 1; q, k,
 * v, out 16-byte aligned.  Sequences of length 0 are allowed (no rows, or no
 * keys).  Device-detected: cu_seqlens not starting at 0, decreasing, not
 * ending at total_q / total_k, or a q length above max_seqlen_q
 * -> VFA_ERR_BAD_SEQLENS, nothing written to out / lse.
 */
vfa_status vfa_varlen_fwd(const void *q, const void *k, const void *v,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          int total_q, int total_k, int max_seqlen_q, int batch,
                          int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                          int causal, int window_left, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, vfa_stream_t stream);

/*
 * vfa_varlen_fwd with q and k given as FP8 E4M3 codes (1 byte each: 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, no infinities), each tensor
 * with one descale factor: element value = descale * code.  v stays bf16.
 * The plan names FP8 kernel configuration types without content; this is
 * the reading taken.  S = q.k is formed by the tensor core's FP8 product
 * (exact products, fp32 accumulation) and scaled by softmax_scale *
 * descale_q * descale_k; everything after S is as in vfa_varlen_fwd.
 *
 * q_fp8        device uint8 [total_q, num_heads, head_dim] E4M3 codes.
 * k_fp8        device uint8 [total_k, num_kv_heads, head_dim] E4M3 codes.
 * descale_q, descale_k  finite, > 0 (else VFA_ERR_INVALID_ARG).
 * Other arguments, outputs, workspace and errors as in vfa_varlen_fwd;
 * head_dim 64, 128 or 256 (else VFA_ERR_UNSUPPORTED).
 */
vfa_status vfa_varlen_fwd_fp8(const void *q_fp8, const void *k_fp8, const void *v,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                              int total_q, int total_k, int max_seqlen_q, int batch,
                              int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                              float descale_q, float descale_k, int causal, int window_left,
                              void *out, float *lse, void *workspace, size_t workspace_bytes,
                              vfa_stream_t stream);

/*
 * vfa_varlen_fwd without a caller workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * code on a real-time or callback thread that must not enter the allocator,
 * runtimes that give kernels a fixed memory plan and forbid other
 * allocations, plugins that only receive their inputs' and outputs' pointers.
 *
 * Same arguments, results and device checks as vfa_varlen_fwd, minus the
 * workspace: the scratch (status word, work list, scheduler records) lives
 * in one 1 MiB array inside the library, which every GPU that loads the
 * library keeps reserved until the process exits.  It allocates nothing and
 * frees nothing.
 *
 * device_status  nullable device int32 [1]: receives the call's status word
 *                (VFA_OK or VFA_ERR_BAD_SEQLENS ...), copied on `stream`.
 *
 * Limits and rules:
 *   - a problem whose vfa_varlen_fwd_workspace_bytes() exceeds 1 MiB returns
 *     VFA_ERR_UNSUPPORTED and enqueues nothing.  That size is exactly
 *     round256(round256(256 + 32 * num_heads * (total_q / 128 + batch))
 *     + 56 * (batch + 1)) bytes (integer division; round256 rounds up to a
 *     multiple of 256): the status word and counters, 32 bytes per work
 *     item, then 14 int32 of scheduler records per sequence;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) and remembers it together with the current CUDA
 *     context; a call under another context (after cudaDeviceReset, or a
 *     thread with a context of its own) looks it up again.  Make such first
 *     calls before any stream capture;
 *   - all calls share the one array: calls whose work can overlap on the GPU
 *     (different streams without ordering) race and give undefined results.
 *     Each call rewrites every scratch word it reads, so stream-ordered calls
 *     are independent.
 */
vfa_status vfa_varlen_fwd_noalloc(const void *q, const void *k, const void *v,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  int total_q, int total_k, int max_seqlen_q, int batch,
                                  int num_heads, int num_kv_heads, int head_dim,
                                  float softmax_scale, int causal, int window_left, void *out,
                                  float *lse, int32_t *device_status, vfa_stream_t stream);

/*
 * The device tile scheduler alone (the first kernel vfa_varlen_fwd runs),
 * writing into caller buffers so the work list can be inspected.
 *
 * A tile is q tile i (local rows [i*block_q, min(Lq_b, (i+1)*block_q))) of
 * sequence b and head h; it visits the key tiles [first, end) that hold a
 * key its rows may see, and its cost is end - first.  Without a window
 * first = 0 and end = ceil(Lk_b / block_k), or with a causal mask
 * ceil(clamp(min(Lq_b, (i+1)*block_q) + off, 0, Lk_b) / block_k), off = 0 for
 * causal == 1 and Lk_b - Lq_b for causal == 2; a window (window_left >= 0,
 * as in vfa_varlen_fwd) gives first = floor(max(0, i*block_q + off -
 * window_left) / block_k); a tile that sees no key has first = end = 0.
 * The tiles of one (b, h) stay together; groups are ordered by their
 * largest cost, then total cost (descending), then (b, h); inside a group
 * by cost descending, then i (with a window: by i descending).  With
 * pair_tiles != 0 two consecutive tiles of a group form one item (what
 * vfa_varlen_fwd uses for head_dim <= 128); otherwise each tile is one
 * item.  Each item is eight int32: (b, i_a, h, end_a, i_b, end_b, first_a,
 * first_b), with i_b = -1 and end_b = first_b = 0 when the second slot is
 * empty.  Sequences with Lq_b == 0 give no items.
 *
 * block_k must be a power of two and block_q a multiple of block_k
 * (VFA_ERR_UNSUPPORTED otherwise); vfa_varlen_fwd_tile_shape() only returns
 * such shapes.
 *
 * items        device int32 [items_capacity, 8] (output).
 * n_items      device int32 [1] (output): number of items written.
 * status       device int32 [1] (output): VFA_OK or a device-detected code.
 * scratch      device scratch of vfa_varlen_fwd_workspace_bytes() bytes,
 *              8-byte aligned.
 */
vfa_status vfa_varlen_schedule(const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                               int total_q, int total_k, int max_seqlen_q, int batch,
                               int num_heads, int block_q, int block_k, int causal,
                               int window_left, int pair_tiles, int32_t *items,
                               int items_capacity,
                               int32_t *n_items, int32_t *status, void *scratch,
                               size_t scratch_bytes, vfa_stream_t stream);

/*
 * Gradients of vfa_varlen_fwd: dq, dk, dv for an upstream gradient dout.
 *
 * The pages name a varlen backward without defining it; this computes the
 * exact derivative of the forward's definition (same masks, head grouping
 * and window): with P = exp(scale * q.k - lse) over a row's visible keys,
 * dP = dout . v, Delta = sum_d dout * out and dS = P * (dP - Delta):
 *   dv[j] = sum_i P_ij dout_i,  dk[j] = scale * sum_i dS_ij q_i,
 *   dq[i] = scale * sum_j dS_ij k_j,
 * with dk, dv of a kv head summed over its query heads.  P and dS are
 * rounded to bf16 for the products (fp32 accumulation), as the forward's P.
 *
 * q, out, dout  device bf16 [total_q, num_heads, head_dim] (out and lse are
 *               the forward's results for these q, k, v).
 * k, v          device bf16 [total_k, num_kv_heads, head_dim].
 * lse           device f32 [total_q, num_heads], natural log (-FLT_MAX for
 *               rows without visible keys, which get dq = 0).
 * cu_seqlens_q/k, total_q/k, batch, num_heads, num_kv_heads, softmax_scale,
 * causal, window_left: as in vfa_varlen_fwd (softmax_scale must be > 0).
 * dq            device bf16 [total_q, num_heads, head_dim] (output).
 * dk, dv        device bf16 [total_k, num_kv_heads, head_dim] (output; keys
 *               no query sees get 0).
 * workspace     device scratch of vfa_varlen_bwd_workspace_bytes() bytes,
 *               256-byte aligned (status word, per-sequence key-tile and
 *               q-tile starts, Delta = rowsum(dout * out)); calls sharing it
 *               must be stream-ordered.  Its first int32 is the device status word
 *               (read with vfa_read_status): VFA_ERR_BAD_SEQLENS for invalid
 *               cu_seqlens (nothing written), VFA_ERR_TIMEOUT if a bounded
 *               wait expired.
 *
 * Supported: head_dim 64, 128 or 256 (others: VFA_ERR_UNSUPPORTED); 16-byte
 * aligned tensors.  No gradient is accumulated with atomics: dk and dv are
 * summed per key tile and dq per query tile in a fixed order, so the three
 * are bit-identical from run to run.
 */
size_t vfa_varlen_bwd_workspace_bytes(int batch, int total_q, int num_heads, int head_dim);

vfa_status vfa_varlen_bwd(const void *q, const void *k, const void *v, const void *out,
                          const void *dout, const float *lse, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, int total_q, int total_k, int batch,
                          int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                          int causal, int window_left, void *dq, void *dk, void *dv,
                          void *workspace, size_t workspace_bytes, vfa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Paged GQA decode                                                          */
/* ------------------------------------------------------------------------ */

/*
 * AttnState::new of "attention_ref.rs" (spark_storage): m = -inf, l = 0,
 * o = 0.
 *
 * m, l   device f32 [num_seqs, num_q_heads]; o device f32 [num_seqs,
 *        num_q_heads, head_dim].  device_status (nullable) device int32 [1] is
 *        set to VFA_OK.
 */
vfa_status vfa_paged_decode_init(float *m, float *l, float *o, int num_seqs, int num_q_heads,
                                 int head_dim, int32_t *device_status, vfa_stream_t stream);

/*
 * One tile update, step_tile_ref of "attention_ref.rs": for every sequence s
 * and q head qh (kv head kh = qh / (num_q_heads / num_kv_heads)) the state
 * (m, l, o) absorbs every one of the block_size tokens of every block id
 * tile_blocks[s, 0:tile_block_counts[s]]; logits are (q . k) / sqrt(head_dim).
 * After any sequence of steps the state satisfies m = max logit, l = sum
 * exp(logit - m), o = sum exp(logit - m) v over all tokens absorbed so far
 * (m is in natural-log units).  Each KV block is read once per kv head group.
 *
 * Two arguments extend the page's step (which always takes whole blocks and
 * 1/sqrt(head_dim)) for contexts that end inside their last block and for
 * other scales: with tile_token_counts the step absorbs only the first
 * tile_token_counts[s] tokens of sequence s's listed blocks, in list order
 * (blocks holding none of them are not read); softmax_scale > 0 replaces
 * 1/sqrt(head_dim).
 *
 * q                 device bf16 [num_seqs, num_q_heads, head_dim].
 * k_pool, v_pool    device bf16 [num_blocks, block_size, num_kv_heads, head_dim].
 * tile_blocks       device int32 [num_seqs, tile_capacity]: physical block ids.
 * tile_block_counts device int32 [num_seqs]: entries used per row (0 = no-op).
 * tile_token_counts nullable device int32 [num_seqs]: tokens to absorb, in
 *                   [0, tile_block_counts[s] * block_size] (0 = no-op); NULL
 *                   = every token of every listed block.
 * softmax_scale     logit scale; <= 0 means 1/sqrt(head_dim); NaN or inf is
 *                   VFA_ERR_INVALID_ARG.
 * m, l, o           the state (in/out), as in vfa_paged_decode_init.
 * device_status     nullable device int32 [1]: a count outside
 *                   [0, tile_capacity], a token count outside its range or a
 *                   block id outside [0, num_blocks) stores VFA_ERR_BAD_BLOCK
 *                   here (first error wins) and that sequence's state is left
 *                   unchanged for this step.
 *
 * Supported: head_dim in {64, 128, 256}; block_size == 16;
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}; num_blocks <= 2^26.
 */
vfa_status vfa_paged_decode_step(const void *q, const void *k_pool, const void *v_pool,
                                 int num_blocks, const int32_t *tile_blocks,
                                 const int32_t *tile_block_counts,
                                 const int32_t *tile_token_counts, int tile_capacity,
                                 int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size, float softmax_scale, float *m,
                                 float *l, float *o, int32_t *device_status,
                                 vfa_stream_t stream);

/*
 * vfa_paged_decode_step with each (sequence, kv head) tile cut into
 * num_splits contiguous runs of its blocks, one CTA per run, so a batch of
 * few sequences with long tiles still spreads over every SM.  The result
 * is the same state update: "attention_ref.rs" (file header) requires a
 * tile's fragmentation to give the single-shot result, and the runs are
 * merged with the same rule the step applies across tiles (m = max of the
 * parts, l and o rescaled by exp(m_part - m) and summed).
 *
 * Each run's CTA writes its partial (m, l, o) to `workspace` and takes a
 * ticket (one atomic add); the last CTA of a (sequence, kv head) merges
 * every run with the incoming state, writes (m, l, o) and sets the ticket
 * back to zero.  No CTA waits for another.
 *
 * Arguments, results and device checks as in vfa_paged_decode_step, plus:
 * num_splits     runs per tile, 1 ..  1024 (1 = vfa_paged_decode_step;
 *                vfa_paged_decode_split_count suggests one); runs past a
 *                tile's last block are empty.
 * workspace      device scratch of vfa_paged_decode_split_workspace_bytes()
 *                bytes, 256-byte aligned, ignored when num_splits == 1.  It
 *                must hold zeros before its first use (e.g. cleared when
 *                allocated); every call leaves it that way.  Calls sharing
 *                one workspace must be stream-ordered.
 */
vfa_status vfa_paged_decode_step_split(const void *q, const void *k_pool, const void *v_pool,
                                       int num_blocks, const int32_t *tile_blocks,
                                       const int32_t *tile_block_counts,
                                       const int32_t *tile_token_counts, int tile_capacity,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float softmax_scale,
                                       float *m, float *l, float *o, int32_t *device_status,
                                       int num_splits, void *workspace, size_t workspace_bytes,
                                       vfa_stream_t stream);

/*
 * Workspace bytes of vfa_paged_decode_step_split: one ticket per (sequence,
 * kv head) and (head_dim + 2) floats per (sequence, q head, run).  0 for
 * unsupported sizes.
 */
size_t vfa_paged_decode_split_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, int num_splits);

/*
 * A run count for vfa_paged_decode_step_split on the current device: about
 * four CTAs per SM over num_seqs * num_kv_heads rows, with runs of at least
 * eight blocks of a tile_capacity-block tile.
 */
vfa_status vfa_paged_decode_split_count(int num_seqs, int num_kv_heads, int tile_capacity,
                                        int *num_splits);

/*
 * finalize_ref of "attention_ref.rs": out = bf16(o * (l > 0 ? 1 / l : 0)),
 * round to nearest even.  l: device f32 [num_seqs, num_q_heads]; o: device
 * f32 [num_seqs, num_q_heads, head_dim]; out: device bf16, same shape as o.
 */
vfa_status vfa_paged_decode_finalize(const float *l, const float *o, int num_seqs,
                                     int num_q_heads, int head_dim, void *out,
                                     vfa_stream_t stream);

/*
 * Test hook for the block-table gather of vfa_paged_decode_step: runs the
 * same device address computation and writes, for every sequence s, listed
 * block b < count_s, token t and kv head kh, the K and V rows it reads into
 * k_out / v_out (device bf16 [num_seqs, tile_capacity, block_size,
 * num_kv_heads, head_dim]); unlisted slots are left untouched.  Errors as in
 * vfa_paged_decode_step.
 */
vfa_status vfa_debug_paged_gather(const void *k_pool, const void *v_pool, int num_blocks,
                                  const int32_t *tile_blocks, const int32_t *tile_block_counts,
                                  int tile_capacity, int num_seqs, int num_kv_heads,
                                  int head_dim, int block_size, void *k_out, void *v_out,
                                  int32_t *device_status, vfa_stream_t stream);

/*
 * Test hook for the bounded waits of every kernel in this library (no
 * counterpart on the pages): one CTA waits on a barrier that nothing
 * arrives on, gives up after the same limit as the pipeline waits (1 s),
 * stores VFA_ERR_TIMEOUT in device_status (first error wins) and exits; the
 * context stays usable.  device_status: device int32 [1], not NULL.
 */
vfa_status vfa_debug_bounded_wait(int32_t *device_status, vfa_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * Waits for `stream`, then copies the device int32 at `device_status_word`
 * (the first word of a vfa_varlen_fwd workspace, or a decode device_status)
 * to *host_status.
 */
vfa_status vfa_read_status(const void *device_status_word, vfa_stream_t stream,
                           int32_t *host_status);

#ifdef __cplusplus
}
#endif

#endif /* VFA_H */
