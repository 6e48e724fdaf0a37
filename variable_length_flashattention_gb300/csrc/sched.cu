// sched.cu -- device-side varlen tile scheduler.
//
// The plan's kernel ("Varlen Flash Attention Implementation Plan", Task 1
// Step 1) gives each block a global q-tile start and finds its sequence by a
// linear scan over cu_seqlens_q; that covers only part of the tokens.  Here
// one CTA turns cu_seqlens into an explicit work list instead:
//   * one item per (sequence b, local q tile i, head h) with Lq_b > 0;
//   * cost = number of key tiles the item visits (fully masked causal tiles
//     are never visited);
//   * order: cost descending (longest-processing-time first, so long
//     sequences start early and the tail is short), ties by (b, i, h).
// It also validates cu_seqlens and max_seqlen_q and reports through the
// status word instead of trapping.
#include "internal.h"

namespace vfa {

namespace {

constexpr int kThreads = 1024;
constexpr int kSmemTiles = 4096;   // tile records kept in shared memory when they fit
constexpr int kSmemHist = 4096;    // cost buckets kept in shared memory when they fit
constexpr size_t kSchedSmem = (3 * kSmemTiles + kSmemHist) * sizeof(int);

__host__ __device__ inline int ceil_div_i(long long a, long long b)
{
    return static_cast<int>((a + b - 1) / b);
}

__host__ __device__ inline int max_tiles(int batch, int total_q, int block_q)
{
    return total_q / block_q + batch;
}

// Exclusive prefix sum of one int per thread over the 1024-thread block.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sums[lane] = w;               // inclusive over warps
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();                       // warp_sums is reused by the next call
    return excl;
}

__global__ void __launch_bounds__(kThreads) schedule_kernel(const SchedArgs a)
{
    extern __shared__ int sm[];
    __shared__ int warp_sums[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x;

    if (tid == 0)
        s_bad = 0;
    __syncthreads();
    if (tid == 0) {
        if (a.cu_q[0] != 0 || a.cu_k[0] != 0 || a.cu_q[a.batch] != a.total_q ||
            a.cu_k[a.batch] != a.total_k)
            s_bad = 1;
    }
    for (int b = tid; b < a.batch; b += kThreads) {
        const long long lq = static_cast<long long>(a.cu_q[b + 1]) - a.cu_q[b];
        const long long lk = static_cast<long long>(a.cu_k[b + 1]) - a.cu_k[b];
        if (lq < 0 || lk < 0 || lq > a.max_seqlen_q)
            s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            *a.n_items = 0;
            *a.status = VFA_ERR_BAD_SEQLENS;
        }
        return;
    }

    // Per-sequence q-tile counts and their exclusive prefix sum.
    int *tile_start = a.scratch;                                 // [batch + 1]
    int carry = 0;
    for (int base = 0; base < a.batch; base += kThreads) {
        const int b = base + tid;
        const int n = b < a.batch ? ceil_div_i(a.cu_q[b + 1] - a.cu_q[b], a.block_q) : 0;
        int total;
        const int ex = block_exclusive_scan(n, warp_sums, &total);
        if (b < a.batch)
            tile_start[b] = carry + ex;
        carry += total;
    }
    const int ntiles = carry;
    if (tid == 0)
        tile_start[a.batch] = ntiles;
    const long long nitems = static_cast<long long>(ntiles) * a.num_heads;
    const int tiles_cap = max_tiles(a.batch, a.total_q, a.block_q);
    const int maxc = ceil_div_i(a.total_k, a.block_k);
    if (nitems > a.item_capacity || ntiles > tiles_cap ||
        (a.batch + 1) + 3LL * tiles_cap + (maxc + 1) > a.scratch_ints) {
        if (tid == 0) {
            *a.n_items = 0;
            *a.status = VFA_ERR_WORKSPACE;
        }
        return;
    }

    const bool tiles_in_smem = ntiles <= kSmemTiles;
    const bool hist_in_smem = maxc + 1 <= kSmemHist;
    int *g_rec = a.scratch + (a.batch + 1);
    int *t_seq = tiles_in_smem ? sm : g_rec;
    int *t_cost = tiles_in_smem ? sm + kSmemTiles : g_rec + tiles_cap;
    int *t_pos = tiles_in_smem ? sm + 2 * kSmemTiles : g_rec + 2 * tiles_cap;
    int *hist = hist_in_smem ? sm + 3 * kSmemTiles : g_rec + 3 * tiles_cap;

    for (int c = tid; c <= maxc; c += kThreads)
        hist[c] = 0;
    __syncthreads();

    // Each tile: its sequence, its cost, and a histogram of costs.
    for (int t = tid; t < ntiles; t += kThreads) {
        int lo = 0, hi = a.batch - 1;              // largest b with tile_start[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        const int i = t - tile_start[b];
        const int lq = a.cu_q[b + 1] - a.cu_q[b];
        const int lk = a.cu_k[b + 1] - a.cu_k[b];
        int cost;
        if (a.causal) {
            const long long last_row_plus_one = min(static_cast<long long>(lq),
                                                    static_cast<long long>(i + 1) * a.block_q);
            cost = ceil_div_i(min(static_cast<long long>(lk), last_row_plus_one), a.block_k);
        } else {
            cost = ceil_div_i(lk, a.block_k);
        }
        t_seq[t] = b;
        t_cost[t] = cost;
        atomicAdd(&hist[cost], 1);
    }
    __syncthreads();

    // Bucket starts in descending cost order: start(c) = #tiles with cost > c.
    carry = 0;
    for (int base = 0; base <= maxc; base += kThreads) {
        const int r = base + tid;
        const int c = maxc - r;
        const int v = r <= maxc ? hist[c] : 0;
        int total;
        const int ex = block_exclusive_scan(v, warp_sums, &total);
        if (r <= maxc)
            hist[c] = carry + ex;
        carry += total;
    }
    __syncthreads();

    // Stable placement: within a bucket, tiles keep their (b, i) order.
    if (tid < 32) {
        const int lane = tid;
        for (int base = 0; base < ntiles; base += 32) {
            const int t = base + lane;
            const bool valid = t < ntiles;
            const int c = valid ? t_cost[t] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, c);
            int start = 0;
            if (valid) {
                start = hist[c];
                t_pos[t] = start + __popc(peers & ((1u << lane) - 1u));
            }
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1)
                hist[c] = start + __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    const int H = a.num_heads;
    for (long long e = tid; e < nitems; e += kThreads) {
        const int t = static_cast<int>(e / H);
        const int h = static_cast<int>(e % H);
        const int b = t_seq[t];
        a.items[static_cast<long long>(t_pos[t]) * H + h] =
            make_int4(b, t - tile_start[b], h, t_cost[t]);
    }
    if (tid == 0) {
        *a.n_items = static_cast<int>(nitems);
        *a.status = VFA_OK;
    }
}

}  // namespace

int schedule_scratch_ints(int batch, int total_q, int total_k, int block_q, int block_k)
{
    return (batch + 1) + 3 * max_tiles(batch, total_q, block_q) + ceil_div_i(total_k, block_k) + 1;
}

cudaError_t launch_schedule(const SchedArgs &a, cudaStream_t stream)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSchedSmem));
        if (e != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    schedule_kernel<<<1, kThreads, kSchedSmem, stream>>>(a);
    return cudaGetLastError();
}

WorkspaceLayout workspace_layout(int batch, int total_q, int total_k, int num_heads,
                                 int block_q, int block_k)
{
    WorkspaceLayout w;
    w.items_offset = 256;
    w.item_capacity = max_tiles(batch, total_q, block_q) * num_heads;
    w.scratch_offset = w.items_offset + static_cast<size_t>(w.item_capacity) * sizeof(int4);
    w.scratch_offset = (w.scratch_offset + 255) & ~static_cast<size_t>(255);
    w.scratch_ints = schedule_scratch_ints(batch, total_q, total_k, block_q, block_k);
    w.total_bytes = w.scratch_offset + static_cast<size_t>(w.scratch_ints) * sizeof(int);
    w.total_bytes = (w.total_bytes + 255) & ~static_cast<size_t>(255);
    return w;
}

}  // namespace vfa
