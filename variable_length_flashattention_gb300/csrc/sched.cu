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
//     work starts first and the tail is short;
//   * in pair mode two consecutive tiles of a group make one item, so one
//     CTA runs both q tiles against each key/value tile it loads.
// It also validates cu_seqlens and max_seqlen_q and reports through the
// status word instead of trapping.
//
// With block_q = r * block_k (r a whole number) and block_k a power of two,
// a causal tile costs clamp((i + 1) * r + e, 0, C), where off = 0 (top-left)
// or Lk - Lq (bottom-right), e = ceil(off / block_k) and C = ceil(clamp(Lq +
// off, 0, Lk) / block_k): zero for the first tiles when off < 0, then rising
// by r per tile until it reaches C.  So a sequence's largest and total cost
// and each tile's rank in its group have closed forms, and the kernel needs
// one pass over the sequences and one over the tiles, with no per-tile
// searches.
//
// A sliding window of W keys (with either causal mode) also hides keys below
// row + off - W.  Tile i then visits key tiles [F(i), c(i)) with F(i) =
// max(0, i * r + g), g = floor((off - W) / block_k), except that the tiles
// from i_z = ceil((Lk - off + W) / block_q) on see no key at all.  Its cost
// c(i) - F(i) rises, stays flat, then falls: the sum is a difference of two
// clamped arithmetic series, the largest cost sits next to the first index
// where the flat part begins, and a group keeps its tiles in i-descending
// order (longest first wherever the keys reach past the last query).
#include "internal.h"

namespace vfa {

namespace {

constexpr int kThreads = 1024;
constexpr int kSmemSeqs = 2048;    // per-sequence records kept in shared memory when they fit
// Per-sequence records in ints: total cost (64-bit, two ints), tile start,
// tile count, cost cap C, offset term e, first tile with a non-zero cost,
// first capped tile, largest cost, rank in group order, rank -> sequence,
// first item / H, window edge term g, tiles before the window's empty tail.
constexpr int kSeqInts = 14;
constexpr size_t kSchedSmem = kSeqInts * kSmemSeqs * sizeof(int);

__host__ __device__ inline int max_tiles(int batch, int total_q, int block_q)
{
    return total_q / block_q + batch;
}

// sum over i in [0, n) of clamp(i * r + a, 0, C), for r >= 1.
__device__ long long sum_lin_clamp(long long n, long long r, long long a, long long C)
{
    if (n <= 0 || C <= 0)
        return 0;
    long long i0 = a > 0 ? 0 : (-a) / r + 1;                 // first positive term
    long long i1 = C - a <= 0 ? 0 : (C - a + r - 1) / r;     // first capped term
    i0 = min(i0, n);
    i1 = min(max(i1, i0), n);
    // (i0 + i1 - 1) (i1 - i0) is even: one factor always is
    const long long rising = r * ((i0 + i1 - 1) * (i1 - i0) / 2) + a * (i1 - i0);
    return rising + (n - i1) * C;
}

__device__ __forceinline__ int floor_div_pow2(long long x, int lb)
{
    return static_cast<int>(x >= 0 ? x >> lb : -((-x + (1ll << lb) - 1) >> lb));
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

    extern __shared__ __align__(16) int sm[];
    __shared__ long long warp_sums[32];
    __shared__ int s_bad, s_nseq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.batch, H = a.num_heads;
    const unsigned bq = static_cast<unsigned>(a.block_q), bk = static_cast<unsigned>(a.block_k);
    const unsigned r = bq / bk;                          // block_q = r * block_k
    const int lbk = __ffs(static_cast<int>(bk)) - 1;    // block_k = 2^lbk
    const int causal = a.causal;                         // 0 none, 1 top-left, 2 bottom-right
    const bool window = causal && a.window_left >= 0;

    const int tiles_cap = max_tiles(B, a.total_q, a.block_q);
    const bool in_smem = B + 1 <= kSmemSeqs;
    if (static_cast<long long>(tiles_cap) * H > a.item_capacity ||
        (!in_smem && static_cast<long long>(kSeqInts) * (B + 1) > a.scratch_ints)) {
        if (tid == 0) {
            *a.n_items = 0;
            *a.status = VFA_ERR_WORKSPACE;
        }
        return;
    }
    const int n = in_smem ? kSmemSeqs : B + 1;
    int *rec = in_smem ? sm : a.scratch;
    long long *seq_total = reinterpret_cast<long long *>(rec);
    int *tile_start = rec + 2 * n;
    int *seq_nt = rec + 3 * n;
    int *seq_cap = rec + 4 * n;
    int *seq_e = rec + 5 * n;
    int *seq_ilo = rec + 6 * n;
    int *seq_ihi = rec + 7 * n;
    int *seq_maxc = rec + 8 * n;
    int *seq_rank = rec + 9 * n;
    int *ord = rec + 10 * n;
    int *seq_first = rec + 11 * n;
    int *seq_g = rec + 12 * n;
    int *seq_n1 = rec + 13 * n;

    if (tid == 0) {
        s_bad = 0;
        s_nseq = 0;
    }
    __syncthreads();
    if (tid == 0 && (a.cu_q[0] != 0 || a.cu_k[0] != 0 || a.cu_q[B] != a.total_q ||
                     a.cu_k[B] != a.total_k))
        s_bad = 1;
    // One pass over the sequences: validation, tile count, cost cap, largest
    // and total cost, and the tile-start prefix sum.
    long long carry = 0;
    for (int base = 0; base < B; base += kThreads) {
        const int b = base + tid;
        int nt = 0;
        if (b < B) {
            const long long lq = static_cast<long long>(a.cu_q[b + 1]) - a.cu_q[b];
            const long long lk = static_cast<long long>(a.cu_k[b + 1]) - a.cu_k[b];
            if (lq < 0 || lk < 0 || lq > a.max_seqlen_q) {
                s_bad = 1;
            } else {
                const unsigned uq = static_cast<unsigned>(lq), uk = static_cast<unsigned>(lk);
                nt = static_cast<int>((uq + bq - 1) / bq);
                int cap, e = 0, i_lo = 0, i_hi = 0;
                long long maxc, total;
                if (!causal) {
                    cap = static_cast<int>((uk + bk - 1) >> lbk);
                    maxc = cap;
                    total = static_cast<long long>(nt) * cap;
                } else {
                    // tile i's last row sees keys 0 .. row + off
                    const long long off = causal == 2 ? lk - lq : 0;
                    const long long m = min(lk, max(0ll, lq + off));
                    cap = static_cast<int>((m + bk - 1) >> lbk);
                    e = off >= 0 ? static_cast<int>((off + bk - 1) >> lbk)
                                 : -static_cast<int>((-off) >> lbk);     // ceil(off / bk)
                    const int ir = static_cast<int>(r);
                    if (cap == 0) {
                        i_lo = i_hi = nt;                  // every tile costs 0
                    } else {
                        // zero-cost tiles: (i + 1) r + e <= 0; capped: (i + 1) r + e >= cap
                        i_lo = e < 0 ? min(nt, (-e) / ir) : 0;
                        i_hi = min(nt, max(0, (cap - e + ir - 1) / ir - 1));
                    }
                    maxc = min(static_cast<long long>(cap),
                               max(0ll, static_cast<long long>(nt) * ir + e));
                    // sum over the rising tiles i_lo .. i_hi - 1 of (i + 1) r + e, plus the capped
                    const long long a0 = i_lo + 1, a1 = i_hi;
                    const long long rising = a1 >= a0 ? (a0 + a1) * (a1 - a0 + 1) / 2 : 0;
                    total = cap > 0 ? ir * rising + static_cast<long long>(e) * (i_hi - i_lo) +
                                          static_cast<long long>(nt - i_hi) * cap
                                    : 0;
                    if (window) {
                        // tile i costs c(i) - max(0, i r + g) below n1, nothing after
                        const int g = floor_div_pow2(off - a.window_left, lbk);
                        const long long iz = (max(0ll, lk - off + a.window_left) + bq - 1) / bq;
                        const int n1 = static_cast<int>(min(static_cast<long long>(nt), iz));
                        const long long ar = ir + e;                 // c(i) = clamp(i r + ar, 0, C)
                        total = sum_lin_clamp(n1, ir, ar, cap) -
                                sum_lin_clamp(n1, ir, g, 1ll << 60);
                        maxc = 0;
                        if (n1 > 0) {
                            // the cost is flat from u = i r = min(-g, C - ar) on; the
                            // largest is at the first index past that point or just before
                            const long long ulo = min(static_cast<long long>(-g), cap - ar);
                            const long long i1 = ulo >= 0 ? (ulo + ir - 1) / ir : -((-ulo) / ir);
                            for (int k = 0; k < 2; ++k) {
                                const long long ic = min(max(i1 - k, 0ll), static_cast<long long>(n1 - 1));
                                const long long ci = min(static_cast<long long>(cap), max(0ll, ic * ir + ar));
                                maxc = max(maxc, ci > 0 ? ci - max(0ll, ic * ir + g) : 0ll);
                            }
                        }
                        seq_g[b] = g;
                        seq_n1[b] = n1;
                    }
                }
                seq_nt[b] = nt;
                seq_cap[b] = cap;
                seq_e[b] = e;
                seq_ilo[b] = i_lo;
                seq_ihi[b] = i_hi;
                seq_maxc[b] = nt > 0 ? static_cast<int>(maxc) : -1;
                seq_total[b] = total;
            }
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
    if (s_bad) {
        if (tid == 0) {
            *a.n_items = 0;
            *a.status = VFA_ERR_BAD_SEQLENS;
        }
        return;
    }

    // Rank of each non-empty sequence in (largest cost desc, total desc, b
    // asc), one warp per sequence.
    for (int b = warp; b < B; b += kThreads / 32) {
        if (seq_nt[b] == 0) {
            if (lane == 0)
                seq_rank[b] = -1;
            continue;
        }
        const int mb = seq_maxc[b];
        const long long tb = seq_total[b];
        int cnt = 0;
        for (int o = lane; o < B; o += 32) {
            const int mo = seq_maxc[o];            // -1 for empty sequences: never ahead
            const long long to = seq_total[o];
            cnt += (mo > mb) || (mo == mb && (to > tb || (to == tb && o < b)));
        }
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (lane == 0) {
            seq_rank[b] = cnt;
            ord[cnt] = b;
            atomicAdd(&s_nseq, 1);
        }
    }
    __syncthreads();
    const int nseq = s_nseq;

    // Items per head of each sequence: its tiles, or its tile pairs; the
    // groups of the sequence at rank k start after those of ranks < k.
    auto units = [&](int nt) { return a.pair ? (nt + 1) / 2 : nt; };
    carry = 0;
    for (int base = 0; base < nseq; base += kThreads) {
        const int k = base + tid;
        const int b = k < nseq ? ord[k] : 0;
        const int u = k < nseq ? units(seq_nt[b]) : 0;
        long long total;
        const long long ex = block_exclusive_scan(u, warp_sums, &total);
        if (k < nseq)
            seq_first[b] = static_cast<int>(carry + ex);     // in units of H items
        carry += total;
    }
    const long long nitems = carry * H;
    __syncthreads();

    // Items, one thread per tile writing all its heads.  Sequence b's groups
    // start at H * seq_first[b], head h's group at + h * units(nt); the
    // tile's rank in its group (cost descending, then i) is i - i_hi for
    // capped tiles (equal cost, i ascending), then the rising tiles with i
    // falling, then the zero-cost tiles with i ascending; it lands in item
    // rank (single) or rank / 2, slot rank % 2 (pairs).
    for (int t = tid; t < ntiles; t += kThreads) {
        int lo = 0, hi = B - 1;                     // largest b with tile_start[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        const int i = t - tile_start[b];
        const int nt = seq_nt[b], cap = seq_cap[b], i_lo = seq_ilo[b], i_hi = seq_ihi[b];
        int c = causal ? min(cap, max(0, (i + 1) * static_cast<int>(r) + seq_e[b])) : cap;
        int f = 0;                                  // first key tile
        int rank;
        if (window) {
            // key tiles [max(0, i r + g), c(i)) below n1; none from n1 on
            if (i < seq_n1[b] && c > 0)
                f = max(0, i * static_cast<int>(r) + seq_g[b]);
            else
                c = 0;
            rank = nt - 1 - i;
        } else {
            rank = i >= i_hi ? i - i_hi
                   : i >= i_lo ? (nt - i_hi) + (i_hi - 1 - i)
                               : (nt - i_lo) + i;
        }
        const int slot = a.pair ? (rank & 1) : 0;
        const int unit = a.pair ? rank >> 1 : rank;
        const int per_head = units(nt);
        const bool alone = !a.pair || rank == nt - 1;
        long long pos = static_cast<long long>(seq_first[b]) * H + unit;
        for (int h = 0; h < H; ++h, pos += per_head) {
            // slot a writes its first key tile into the second int4's z, slot b
            // into w; each slot writes only its own words
            int *w = reinterpret_cast<int *>(a.items + 2 * pos);
            if (slot == 0) {
                a.items[2 * pos] = make_int4(b, i, h, c);
                if (alone)
                    a.items[2 * pos + 1] = make_int4(-1, 0, f, 0);
                else
                    w[6] = f;
            } else {
                w[4] = i;
                w[5] = c;
                w[7] = f;
            }
        }
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
    return kSeqInts * (batch + 1);
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
    w.scratch_offset = w.items_offset + static_cast<size_t>(w.item_capacity) * 2 * sizeof(int4);
    w.scratch_offset = (w.scratch_offset + 255) & ~static_cast<size_t>(255);
    w.scratch_ints = schedule_scratch_ints(batch, total_q, total_k, block_q, block_k);
    w.total_bytes = w.scratch_offset + static_cast<size_t>(w.scratch_ints) * sizeof(int);
    w.total_bytes = (w.total_bytes + 255) & ~static_cast<size_t>(255);
    return w;
}

}  // namespace vfa
