// internal.h -- declarations shared by the host API and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/vfa.h"

namespace vfa {

// Records `message` as the calling thread's vfa_last_error() text; returns st.
vfa_status set_error(vfa_status st, const char *message);

// ------------------------------------------------------------ tile shapes

// Query rows per tile: one tcgen05 M=128 accumulator, one TMEM lane per row.
constexpr int kBlockQ = 128;

__host__ __device__ constexpr int block_k_for(int head_dim)
{
    return head_dim == 256 ? 64 : 128;
}

// ------------------------------------------------------------ workspace

// Layout of the varlen forward workspace (all offsets in bytes):
//   [0]   int32 status word
//   [4]   int32 number of work items
//   [8]   int32 next item to take (the prefill's atomic counter)
//   [256] items[item_capacity], 32 bytes each: int4 (b, i_a, h, end_a),
//         int4 (i_b, end_b, first_a, first_b); slot x visits key tiles
//         [first_x, end_x); i_b = -1 when the second slot is empty
//   then  int32 scheduler scratch
struct WorkspaceLayout {
    size_t items_offset;
    int item_capacity;
    size_t scratch_offset;
    int scratch_ints;
    size_t total_bytes;
};

WorkspaceLayout workspace_layout(int batch, int total_q, int total_k, int num_heads,
                                 int block_q, int block_k);

// ------------------------------------------------------------ scheduler

struct SchedArgs {
    const int32_t *cu_q;
    const int32_t *cu_k;
    int batch, total_q, total_k, max_seqlen_q, num_heads, block_q, block_k;
    int causal;           // 0 none, 1 top-left, 2 bottom-right
    int window_left;      // < 0 none; else keys j >= row + off - window_left only (causal != 0)
    int pair;             // non-zero: two consecutive tiles of a group per item
    int4 *items;          // two int4 per item
    int item_capacity;
    int32_t *n_items;
    int32_t *status;
    int32_t *next_item;   // nullable: the prefill's dynamic-fetch counter, reset to 0
    int32_t *scratch;
    int scratch_ints;
};

cudaError_t launch_schedule(const SchedArgs &a, cudaStream_t stream);

// Number of scheduler scratch ints for these sizes.
int schedule_scratch_ints(int batch, int total_q, int total_k, int block_q, int block_k);

// ------------------------------------------------------------ prefill

struct PrefillArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    CUtensorMap tm_o;     // out: boxes of 32 columns x 1 head x 32 rows, 64-byte swizzle
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int4 *items;    // two int4 per item
    const int32_t *n_items;
    int32_t *next_item;   // atomic counter CTAs take items from (reset by the scheduler)
    int32_t *status;
    void *out;
    float *lse;
    int num_heads;
    int kv_group;         // query heads per kv head: K/V of head h live at h / kv_group
    float scale_log2;     // softmax_scale * log2(e), > 0
    int causal;           // 0 none, 1 top-left, 2 bottom-right
    int window_left;      // < 0 none; else keys j >= row + off - window_left only
    int qk_fp8;           // non-zero: tm_q / tm_k map FP8 E4M3 codes (any supported head_dim)
};

// Whether the forward for `head_dim` runs two q tiles per work item.
__host__ __device__ constexpr bool pairs_for(int head_dim)
{
    return head_dim <= 128;
}

// Dispatches by head_dim: two-q-tile kernel (prefill_pair.cu) for 64 and 128,
// single-tile kernel (prefill.cu) for 256.
cudaError_t launch_prefill(int head_dim, const PrefillArgs &a, int grid, cudaStream_t stream);
cudaError_t launch_prefill_pair(int head_dim, const PrefillArgs &a, int grid,
                                cudaStream_t stream);

// ------------------------------------------------------------ decode

struct DecodeStepArgs {
    const void *q, *k_pool, *v_pool;
    const int32_t *tile_blocks, *tile_block_counts;
    const int32_t *tile_token_counts;   // nullable: every token of every listed block
    float scale_log2;                   // logit scale * log2(e), > 0
    int num_blocks, tile_capacity, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    float *m, *l, *o;
    int32_t *status;      // nullable
    // Split step (num_splits > 1): each (kv head, sequence) tile is cut into
    // num_splits contiguous runs of blocks, one CTA each; a CTA writes its
    // partial state to `part` and the last of a row's CTAs (atomic ticket)
    // merges them into (m, l, o).
    int num_splits;
    float *part;          // [num_seqs, num_kv_heads, num_splits, G, D + 2]
    int32_t *tickets;     // [num_seqs, num_kv_heads], zero between calls
};

// Bytes of the split step's workspace: tickets, then the partial states.
size_t decode_split_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int num_splits);
void decode_split_workspace_carve(void *ws, int num_seqs, int num_kv_heads, DecodeStepArgs *a);

cudaError_t launch_decode_init(float *m, float *l, float *o, int num_seqs, int num_q_heads,
                               int head_dim, int32_t *status, cudaStream_t stream);
// K and V pools as 3-D TMA maps over [num_blocks * block_size tokens,
// num_kv_heads, head_dim] (innermost first: dim, kv head, token); box =
// head_dim x 1 x block_size, no swizzle.
struct DecodeMaps {
    CUtensorMap tm_k, tm_v;
};

cudaError_t launch_decode_step(const DecodeStepArgs &a, const DecodeMaps &maps,
                               cudaStream_t stream);
cudaError_t launch_decode_finalize(const float *l, const float *o, int num_seqs,
                                   int num_q_heads, int head_dim, void *out,
                                   cudaStream_t stream);
cudaError_t launch_decode_gather(const DecodeStepArgs &a, void *k_out, void *v_out,
                                 cudaStream_t stream);

// ------------------------------------------------------------ backward

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;   // boxes of 64 columns x 1 head x bwd_step_rows() rows,
                                            // 128-byte swizzle
    CUtensorMap tm_ks, tm_vs;               // K, V with boxes of bwd_dq_step_rows() rows (the
                                            // dQ kernel's streamed tiles)
    CUtensorMap tm_qs, tm_dos;              // Q, dO with boxes of bwd_kv_step_rows() rows (the
                                            // dK/dV kernel's streamed tiles)
    const int32_t *cu_q;
    const int32_t *cu_k;
    const void *out, *dout;                 // bf16 [total_q, H, D]
    const float *lse;                       // f32 [total_q, H], natural log
    void *dq, *dk, *dv;                     // bf16 outputs
    int32_t *status;                        // workspace: status word
    int32_t *ktile_start;                   // workspace: [batch + 1] first 128-key tile per sequence
    int32_t *qtile_start;                   // workspace: [batch + 1] first 128-query tile per sequence
    float *delta;                           // workspace: [total_q, H]
    int batch, total_q, total_k, num_heads, num_kv_heads;
    float scale, scale_log2;
    int causal, window_left;
};

// Rows the backward streams per step (queries past a key tile, keys past a
// query tile); its TMA maps use boxes of this many rows.
__host__ __device__ constexpr int bwd_step_rows(int head_dim)
{
    return head_dim == 256 ? 32 : 64;
}

// Queries the dK/dV kernel streams per step past a key tile (its TMEM holds
// dK, dV and two buffers of 2 x this many columns); the tm_qs / tm_dos maps
// use boxes of this many rows.
__host__ __device__ constexpr int bwd_kv_step_rows(int head_dim)
{
    return head_dim == 64 ? 96 : bwd_step_rows(head_dim);
}

// Keys the dQ kernel streams per step past a query tile; the tm_ks / tm_vs
// maps use boxes of this many rows.
__host__ __device__ constexpr int bwd_dq_step_rows(int head_dim)
{
    return head_dim == 256 ? 32 : 96;
}

// Workspace bytes of the backward and its split into the BwdArgs pointers.
size_t bwd_workspace_bytes(int batch, int total_q, int num_heads, int head_dim);
void bwd_workspace_split(void *ws, int batch, int total_q, int num_heads, BwdArgs *a);
// prep, Delta, then the persistent dK/dV and dQ kernels (one CTA per SM each,
// taking (key tile, kv head) and (q tile, head) units from atomic counters).
cudaError_t launch_bwd(int head_dim, const BwdArgs &a, int key_tile_bound, int q_tile_bound,
                       int sm_count, cudaStream_t stream);

// ------------------------------------------------------------ test hooks

cudaError_t launch_debug_bounded_wait(int32_t *status, cudaStream_t stream);

}  // namespace vfa
