// sched.cu -- device-side varlen tile scheduler.
//
// The plan's kernel ("Varlen Flash Attention Implementation Plan", Task 1
// Step 1) gives each block a global q-tile start and finds its sequence by a
// linear scan over cu_seqlens_q; that covers only part of the tokens.  Here
// one CTA turns cu_seqlens into an explicit work list instead:
//   * one item per (sequence b, local q tile i, head h) with Lq_b > 0, with
//     cost = number of key tiles it visits (fully masked causal key tiles are
//     never visited);
//   * the items of one (b, h) stay together, so the q tiles that read the
//     same keys and values run at the same time and share them through L2;
//   * groups ordered by largest item cost, then total cost (descending),
//     then (b, h); inside a group by cost descending, then i.  The prefill
//     CTAs take items in this order from an atomic counter, so the longest
//     work starts first and the tail is short.
// It also validates cu_seqlens and max_seqlen_q and reports through the
// status word instead of trapping.
#include "internal.h"

namespace vfa {

namespace {

constexpr int kThreads = 1024;
constexpr int kSmemSeqs = 2048;    // per-sequence records kept in shared memory when they fit
constexpr int kSeqRecords = 6;     // tile start, tile count, largest cost, total/first, rank, order
constexpr size_t kSchedSmem = kSeqRecords * kSmemSeqs * sizeof(int);

__host__ __device__ inline int ceil_div_i(long long a, long long b)
{
    return static_cast<int>((a + b - 1) / b);
}

__host__ __device__ inline int max_tiles(int batch, int total_q, int block_q)
{
    return total_q / block_q + batch;
}

// Key tiles that q tile i of a (lq, lk) sequence visits; non-decreasing in i.
__device__ __forceinline__ int tile_cost(int lq, int lk, int i, int bq, int bk, int causal)
{
    if (!causal)
        return ceil_div_i(lk, bk);
    const long long last_row_plus_one = min(static_cast<long long>(lq), static_cast<long long>(i + 1) * bq);
    return ceil_div_i(min(static_cast<long long>(lk), last_row_plus_one), bk);
}

// First tile index in [0, nt) whose cost is > c (ge = false) or >= c (ge = true).
__device__ __forceinline__ int first_tile_above(int lq, int lk, int nt, int c, bool ge, int bq,
                                                int bk, int causal)
{
    int lo = 0, hi = nt;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int cm = tile_cost(lq, lk, mid, bq, bk, causal);
        if (ge ? (cm >= c) : (cm > c))
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// Exclusive prefix sum of one value per thread over the 1024-thread block.
__device__ long long block_exclusive_scan(long long v, long long *warp_sums, long long *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const long long excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kThreads) schedule_kernel(const SchedArgs a)
{
    // Let the dependent prefill grid start its prologue now; it waits for this
    // grid's completion before it reads anything written here.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    extern __shared__ int sm[];
    __shared__ long long warp_sums[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    const int B = a.batch, H = a.num_heads, bq = a.block_q, bk = a.block_k;

    if (tid == 0)
        s_bad = 0;
    __syncthreads();
    if (tid == 0) {
        if (a.cu_q[0] != 0 || a.cu_k[0] != 0 || a.cu_q[B] != a.total_q || a.cu_k[B] != a.total_k)
            s_bad = 1;
    }
    for (int b = tid; b < B; b += kThreads) {
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

    const int tiles_cap = max_tiles(B, a.total_q, bq);
    const long long need = static_cast<long long>(kSeqRecords) * (B + 1);
    if (static_cast<long long>(tiles_cap) * H > a.item_capacity || need > a.scratch_ints) {
        if (tid == 0) {
            *a.n_items = 0;
            *a.status = VFA_ERR_WORKSPACE;
        }
        return;
    }
    // Per-sequence records: tile start, tile count, largest cost, total cost
    // (later: first item / H), rank in group order, and the rank -> sequence order.
    const bool seqs_in_smem = B + 1 <= kSmemSeqs;
    int *g = a.scratch;
    int *tile_start = seqs_in_smem ? sm : g;
    int *seq_nt = seqs_in_smem ? sm + kSmemSeqs : g + (B + 1);
    int *seq_maxc = seqs_in_smem ? sm + 2 * kSmemSeqs : g + 2 * (B + 1);
    int *seq_total = seqs_in_smem ? sm + 3 * kSmemSeqs : g + 3 * (B + 1);
    int *seq_rank = seqs_in_smem ? sm + 4 * kSmemSeqs : g + 4 * (B + 1);
    int *seq_first = seq_total;      // reused once the ranks are known (as item offsets / H)

    // Tile counts, largest cost (the last tile's: costs never decrease in i),
    // and the tile-start prefix sum.
    long long carry = 0;
    for (int base = 0; base < B; base += kThreads) {
        const int b = base + tid;
        int nt = 0;
        if (b < B) {
            const int lq = a.cu_q[b + 1] - a.cu_q[b];
            const int lk = a.cu_k[b + 1] - a.cu_k[b];
            nt = ceil_div_i(lq, bq);
            seq_nt[b] = nt;
            seq_maxc[b] = nt > 0 ? tile_cost(lq, lk, nt - 1, bq, bk, a.causal) : -1;
            seq_total[b] = 0;
        }
        long long total;
        const long long ex = block_exclusive_scan(nt, warp_sums, &total);
        if (b < B)
            tile_start[b] = static_cast<int>(carry + ex);
        carry += total;
    }
    const int ntiles = static_cast<int>(carry);
    if (tid == 0)
        tile_start[B] = ntiles;
    __syncthreads();

    // Total cost per sequence.
    for (int t = tid; t < ntiles; t += kThreads) {
        int lo = 0, hi = B - 1;                     // largest b with tile_start[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int lq = a.cu_q[lo + 1] - a.cu_q[lo];
        const int lk = a.cu_k[lo + 1] - a.cu_k[lo];
        atomicAdd(&seq_total[lo], tile_cost(lq, lk, t - tile_start[lo], bq, bk, a.causal));
    }
    __syncthreads();

    // Rank of each non-empty sequence in (largest cost desc, total desc, b asc).
    for (int b = tid; b < B; b += kThreads) {
        if (seq_nt[b] == 0) {
            seq_rank[b] = -1;
            continue;
        }
        const int mb = seq_maxc[b], tb = seq_total[b];
        int r = 0;
        for (int o = 0; o < B; ++o) {
            if (seq_nt[o] == 0)
                continue;
            const int mo = seq_maxc[o], to = seq_total[o];
            r += (mo > mb) || (mo == mb && (to > tb || (to == tb && o < b)));
        }
        seq_rank[b] = r;
    }
    __syncthreads();

    // Items before each sequence in rank order: a scan over ranks.
    int *ord = seqs_in_smem ? sm + 5 * kSmemSeqs : g + 5 * (B + 1);
    for (int b = tid; b < B; b += kThreads)
        if (seq_rank[b] >= 0)
            ord[seq_rank[b]] = b;
    __syncthreads();
    int nseq = 0;
    {
        // number of non-empty sequences
        long long total;
        int cnt = 0;
        for (int b = tid; b < B; b += kThreads)
            cnt += seq_nt[b] > 0;
        block_exclusive_scan(cnt, warp_sums, &total);
        nseq = static_cast<int>(total);
    }
    carry = 0;
    for (int base = 0; base < nseq; base += kThreads) {
        const int r = base + tid;
        const int b = r < nseq ? ord[r] : 0;
        const int n = r < nseq ? seq_nt[b] : 0;
        long long total;
        const long long ex = block_exclusive_scan(n, warp_sums, &total);
        if (r < nseq)
            seq_first[b] = static_cast<int>(carry + ex);     // in units of H items
        carry += total;
    }
    __syncthreads();

    // Items: sequence b's groups start at H * seq_first[b]; head h's group at
    // + h * nt; the tile's place in its group is its rank by (cost desc, i asc).
    const long long nitems = static_cast<long long>(ntiles) * H;
    for (long long e = tid; e < nitems; e += kThreads) {
        const int t = static_cast<int>(e / H);
        const int h = static_cast<int>(e % H);
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        const int i = t - tile_start[b];
        const int nt = seq_nt[b];
        const int lq = a.cu_q[b + 1] - a.cu_q[b];
        const int lk = a.cu_k[b + 1] - a.cu_k[b];
        const int c = tile_cost(lq, lk, i, bq, bk, a.causal);
        const int above = nt - first_tile_above(lq, lk, nt, c, false, bq, bk, a.causal);
        const int before_equal = i - first_tile_above(lq, lk, nt, c, true, bq, bk, a.causal);
        const long long pos = static_cast<long long>(seq_first[b]) * H +
                              static_cast<long long>(h) * nt + above + before_equal;
        a.items[pos] = make_int4(b, i, h, c);
    }
    if (tid == 0) {
        *a.n_items = static_cast<int>(nitems);
        if (a.next_item)
            *a.next_item = 0;
        *a.status = VFA_OK;
    }
}

}  // namespace

int schedule_scratch_ints(int batch, int total_q, int total_k, int block_q, int block_k)
{
    (void)total_q;
    (void)total_k;
    (void)block_q;
    (void)block_k;
    return kSeqRecords * (batch + 1);
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
