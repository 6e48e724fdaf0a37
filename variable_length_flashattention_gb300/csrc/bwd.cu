// bwd.cu -- variable-length attention backward on sm_103a (head_dim 64, 128,
// 256).
//
// Gradients of the forward (scaled scores, causal / bottom-right / sliding-
// window masks on local positions, softmax over the visible keys) for an
// upstream gradient dO, given the forward's out and natural-log lse.  With
// P = exp(scale * q.k - lse), dP = dO V^T, Delta = rowsum(dO * out) and
// dS = P * (dP - Delta):
//   dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K.
//
// Four kernels, none of them with atomics, so every gradient is
// deterministic:
//   * bwd_prep: one CTA validates cu_seqlens and writes each sequence's first
//     global key tile and first global q tile (prefix sums of
//     ceil(L / 128));
//   * bwd_delta: Delta[t, h] = sum_d dO * out, one warp per (token, head);
//   * the dK/dV kernel (bwd_main_kernel<D, false>): for each 128-key tile and
//     kv head -- at head_dim 256 each column half of dK and dV -- K and V
//     stay in shared memory; the query rows that see a key of the tile stream
//     past in steps of STEP rows (64; 32 at head_dim 256), every query head of
//     the group, Q and dO through a TMA ring.  Per step the tensor core forms
//     S^T = K Q^T and dP^T = V dO^T into one of two TMEM buffers; eight warps
//     turn them into P^T and dS^T (bf16, written back over the columns they
//     read), and the tensor core accumulates dV += P^T dO and dK += dS^T Q in
//     TMEM with both A operands read from TMEM.  With two buffers the next
//     step's S^T / dP^T run on the tensor core while this step's are being
//     exponentiated;
//   * the dQ kernel (bwd_main_kernel<D, true>): for each 128-query tile and
//     head, the same with the roles swapped: Q, dO stay, K and V stream past
//     in blocks of STEP keys (96; 32 at head_dim 256, through their own TMA
//     maps with boxes of that height); S = Q K^T, dP = dO V^T into two TMEM
//     buffers, dS (bf16, over dP) and dQ += dS K in TMEM.  dQ leaves as bf16
//     once, so no fp32 sum and no second pass exist.  It is launched with
//     programmatic dependent launch and starts on the SMs the dK/dV kernel's
//     CTAs leave (it reads nothing that kernel writes).
// Both are persistent: one CTA per SM takes (tile, head) units from an atomic
// counter, and consecutive units overlap (the next unit's own tiles load and
// its first score products run while the current one finishes).  dK, dV and
// dQ leave through a per-warp shared-memory stage.
// The math warps evaluate masks only on steps that need them, as one
// interval of visible columns per thread.  Every wait is bounded; on expiry
// the CTA records VFA_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and
// exits.
#include <algorithm>
#include <cfloat>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

constexpr int kOwn = 128;          // rows of a CTA's own tile (keys, resp. queries)
constexpr int kMathWarps = 8;      // four TMEM lane quarters x two column halves
constexpr int kFirstMathWarp = 4;
constexpr int kMathThreads = kMathWarps * 32;
constexpr int kThreads = (kFirstMathWarp + kMathWarps) * 32;   // + TMA, MMA, two idle warps
constexpr int kPrepThreads = 1024;
constexpr uint32_t kEpiStage = 32 * 64;    // per math warp: 32 rows x 32 bf16 columns of output
constexpr float kLog2e = 1.4426950408889634f;

// Shapes per head_dim and kernel (DQ: the dQ kernel).  STEP rows (queries,
// resp. keys) stream past per step, as many as TMEM holds two buffers of:
// 96 keys past a query tile (dQ + 2 x (2 x 96) columns at head_dim 128), 64
// queries past a key tile at head_dim 128 (dK, dV and 2 x (2 x 64)) and 96
// at head_dim 64; N = 96 score products run at 56.9 cycles against 48.9 at
// N = 64 for 1.5x the work.  32 either way at head_dim 256, so that the own
// tiles and a two-stage ring fit shared memory.  The dK/dV kernel splits dK and dV into DSPLIT column
// halves, one CTA each (at head_dim 256 the two accumulators would fill TMEM
// alone).
template <int D, bool DQ>
struct BwdCfg {
    static constexpr int DB = D / 64;                       // 128-byte column blocks per row
    static constexpr int STEP = DQ ? bwd_dq_step_rows(D) : bwd_kv_step_rows(D);   // TMA box height
    static constexpr int OWN_BOX = bwd_step_rows(D);        // box height of the own-tile maps
    static constexpr int NCH = STEP / 32;                   // 32-column chunks per step
    static constexpr int DSPLIT = D == 256 ? 2 : 1;
    static constexpr int DKV = D / DSPLIT;                  // dK / dV columns per CTA
    static constexpr uint32_t OWN_BYTES = kOwn * D * 2;     // a 128-row tile
    static constexpr uint32_t STEP_BYTES = STEP * D * 2;    // a STEP-row tile
    // streamed-tile ring stages (three 96-key stages at head_dim 128 fill
    // shared memory)
    static constexpr int NSTAGE = D == 256 ? 2 : (DQ && STEP == 96 && D == 128 ? 3 : 4);
    static constexpr uint32_t STAGE_BYTES = 2 * STEP_BYTES; // (Q, dO) or (K, V)
    // per math warp: -lse log2(e) and -Delta of a step's query columns (the
    // dK/dV kernel only; the dQ kernel keeps its rows' in registers)
    static constexpr uint32_t STAT_BYTES = DQ ? 0 : 256 * NCH;
    // TMEM.  dK/dV kernel: dV, dK (DKV columns each), then two buffers of S^T
    // (STEP columns) + dP^T (STEP).  dQ kernel: dQ (D), then the two buffers.
    static constexpr uint32_t COL_DV = 0, COL_DK = DKV, KV_BUF = 2 * DKV;
    static constexpr uint32_t COL_DQ = 0, Q_BUF = D;
    static constexpr uint32_t BUF_STRIDE = 2 * STEP;
    static constexpr uint32_t TMEM_COLS = 512;
    // ring full / empty per stage; s_full, p_full, unit_full, unit_empty per
    // buffer; own_full, own_empty, acc_done, epi_done, drain
    static constexpr int NUM_BARS = 2 * NSTAGE + 8 + 5;
    static constexpr size_t SMEM = 1024 + 2 * OWN_BYTES + NSTAGE * STAGE_BYTES +
                                   kMathWarps * (STAT_BYTES + kEpiStage) + NUM_BARS * 8 + 64;
    // S^T / dP^T (keys x STEP queries) and S / dP (queries x STEP keys): both K-major
    static constexpr uint32_t IDESC_T = idesc_bf16_f32(kOwn, STEP, false, false);
    // dV, dK (DKV columns) and dQ (D columns): A from TMEM, B (dO, Q or K rows) MN-major
    static constexpr uint32_t IDESC_KV = idesc_bf16_f32(kOwn, DKV, false, true);
    static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(kOwn, D, false, true);
    static_assert((DQ ? Q_BUF : KV_BUF) + 2 * BUF_STRIDE <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(STEP % 32 == 0 && STEP <= 256 && kOwn % OWN_BOX == 0, "step shape");
};

// ------------------------------------------------------------ prep

// Exclusive prefix sum over blockDim.x-wide chunks of per-sequence counts;
// out[b] = sum of count(b') for b' < b, out[B] = the total.
template <typename CountFn>
__device__ void block_prefix(int B, int32_t *out, int *warp_sums, CountFn count)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    for (int base = 0; base < B; base += kPrepThreads) {
        const int b = base + tid;
        const int nt = b < B ? count(b) : 0;
        int x = nt;
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
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int excl = x - nt + (warp > 0 ? warp_sums[warp - 1] : 0);
        if (b < B)
            out[b] = carry + excl;
        carry += warp_sums[31];
        __syncthreads();
    }
    if (tid == 0)
        out[B] = carry;
}

__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const BwdArgs a)
{
    __shared__ int warp_sums[32];
    __shared__ int s_bad;
    const int B = a.batch;
    if (threadIdx.x == 0)
        s_bad = (a.cu_q[0] != 0 || a.cu_k[0] != 0 || a.cu_q[B] != a.total_q ||
                 a.cu_k[B] != a.total_k);
    __syncthreads();
    block_prefix(B, a.ktile_start, warp_sums, [&](int b) {
        const int lq = a.cu_q[b + 1] - a.cu_q[b], lk = a.cu_k[b + 1] - a.cu_k[b];
        if (lq < 0 || lk < 0) {
            s_bad = 1;
            return 0;
        }
        return (lk + kOwn - 1) / kOwn;
    });
    block_prefix(B, a.qtile_start, warp_sums, [&](int b) {
        const int lq = a.cu_q[b + 1] - a.cu_q[b];
        return lq > 0 ? (lq + kOwn - 1) / kOwn : 0;
    });
    __syncthreads();
    if (threadIdx.x == 0) {
        a.status[1] = 0;                 // unit counters of the two main kernels
        a.status[2] = 0;
        *a.status = s_bad ? VFA_ERR_BAD_SEQLENS : VFA_OK;
    }
}

// ------------------------------------------------------------ Delta

template <int D>
__global__ void bwd_delta_kernel(const BwdArgs a)
{
    if (*a.status != VFA_OK)
        return;
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(a.total_q) * a.num_heads;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const __nv_bfloat16 *o = static_cast<const __nv_bfloat16 *>(a.out);
    const __nv_bfloat16 *g = static_cast<const __nv_bfloat16 *>(a.dout);
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         r < rows; r += warps) {
        float s = 0.f;
#pragma unroll
        for (int d = lane * 2; d < D; d += 64) {
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(o + r * D + d);
            const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162 *>(g + r * D + d);
            s += __bfloat162float(x.x) * __bfloat162float(y.x) +
                 __bfloat162float(x.y) * __bfloat162float(y.y);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o2);
        if (lane == 0)
            a.delta[r] = s;
    }
}

// ------------------------------------------------------------ shared pieces

// Largest b with start[b] <= gt (start is a non-decreasing prefix sum).
__device__ __forceinline__ int owner_of(const int32_t *start, int B, int gt)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (start[mid] <= gt)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// The visible part of (at most 32) consecutive columns, [lo, hi) (empty when hi <= lo),
// clamped to [-1, 33] so it fits an int.
__device__ __forceinline__ int clamp_col(long long x)
{
    return static_cast<int>(x < -1 ? -1 : (x > 33 ? 33 : x));
}

// Key j's visible queries among i_base, i_base + 1, ... (the dK/dV kernel's
// columns): i < Lq, and i >= j - off (causal), i <= j - off + window_left.
__device__ __forceinline__ void key_row_span(long long j, long long i_base, int lk, int lq,
                                             int causal, int wl, long long off, int *lo, int *hi)
{
    long long l = causal ? j - off - i_base : 0;
    long long h = lq - i_base;
    if (wl >= 0)
        h = min(h, j - off + wl - i_base + 1);
    if (j >= lk)
        h = l;
    *lo = clamp_col(l);
    *hi = clamp_col(h);
}

// Query i's visible keys among j_base, j_base + 1, ... (the dQ kernel's
// columns): j < Lk, and j <= i + off (causal), j >= i + off - window_left.
__device__ __forceinline__ void query_row_span(long long i, long long j_base, int lk, int lq,
                                               int causal, int wl, long long off, int *lo,
                                               int *hi)
{
    long long l = (causal && wl >= 0) ? i + off - wl - j_base : 0;
    long long h = lk - j_base;
    if (causal)
        h = min(h, i + off - j_base + 1);
    if (i >= lq)
        h = l;
    *lo = clamp_col(l);
    *hi = clamp_col(h);
}

// P^T and dS^T of this thread's key row over its NC query columns: p =
// 2^(s scale_log2 + nl) (0 outside the visible columns [lo, hi) when MASK)
// and ds = p (dp + nd), with nl = -lse log2(e) and nd = -Delta of each column
// read from shared memory (NC floats each at wstat, wstat + 128).
template <bool MASK, int NC>
__device__ __forceinline__ void key_row_grads(const uint32_t (&sr)[NC], const uint32_t (&dr)[NC],
                                              float scale_log2, uint32_t wstat, int lo, int hi,
                                              uint32_t (&pk)[NC / 2], uint32_t (&dk2)[NC / 2])
{
    const float2 c2 = make_float2(scale_log2, scale_log2);
#pragma unroll
    for (int e = 0; e < NC; e += 4) {
        const uint4 nl4 = ld_shared_v4(wstat + e * 4);
        const uint4 nd4 = ld_shared_v4(wstat + 128 + e * 4);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const uint32_t nla = u ? nl4.z : nl4.x, nlb = u ? nl4.w : nl4.y;
            const uint32_t nda = u ? nd4.z : nd4.x, ndb = u ? nd4.w : nd4.y;
            const float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[e + u]),
                                                    __uint_as_float(sr[e + u + 1])),
                                        c2, make_float2(__uint_as_float(nla),
                                                        __uint_as_float(nlb)));
            float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
            if (MASK) {
                p0 = (e + u >= lo && e + u < hi) ? p0 : 0.f;
                p1 = (e + u + 1 >= lo && e + u + 1 < hi) ? p1 : 0.f;
            }
            const float2 g = __fadd2_rn(make_float2(__uint_as_float(dr[e + u]),
                                                    __uint_as_float(dr[e + u + 1])),
                                        make_float2(__uint_as_float(nda), __uint_as_float(ndb)));
            const float2 ds = __fmul2_rn(make_float2(p0, p1), g);
            pk[(e + u) >> 1] = pack_bf16x2(p0, p1);
            dk2[(e + u) >> 1] = pack_bf16x2(ds.x, ds.y);
        }
    }
}

// dS of this thread's query row over its NC key columns: p = 2^(s
// scale_log2 + nl) (0 outside [lo, hi) when MASK), ds = p (dp + nd) with the
// row's nl = -lse log2(e) and nd = -Delta.
template <bool MASK, int NC>
__device__ __forceinline__ void query_row_grads(const uint32_t (&sr)[NC], const uint32_t (&dr)[NC],
                                                float scale_log2, float nl, float nd, int lo,
                                                int hi, uint32_t (&dk2)[NC / 2])
{
    const float2 c2 = make_float2(scale_log2, scale_log2);
    const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
#pragma unroll
    for (int e = 0; e < NC; e += 2) {
        const float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                    c2, nl2);
        float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
        if (MASK) {
            p0 = (e >= lo && e < hi) ? p0 : 0.f;
            p1 = (e + 1 >= lo && e + 1 < hi) ? p1 : 0.f;
        }
        const float2 g = __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                    nd2);
        const float2 ds = __fmul2_rn(make_float2(p0, p1), g);
        dk2[e >> 1] = pack_bf16x2(ds.x, ds.y);
    }
}

// Loads a tile of `rows` rows (a multiple of the map's box height BOX) of
// every 64-column block of row `row0`, head `head` into a 128-byte-swizzled
// buffer holding `rows` rows per column block.
template <int DB, int BOX>
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                          int head, int row0, int rows)
{
    for (int db = 0; db < DB; ++db)
        for (int r = 0; r < rows; r += BOX)
            tma_load_3d(dst + db * (rows * 128) + r * 128, map, bar, db * 64, head, row0 + r);
}

// S (or S^T) = A B^T over K = D for A a 128-row operand and B a STEP-row
// operand, both K-major in 128-byte-swizzled column blocks.
template <int D, int STEP>
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, uint32_t a_buf, uint32_t b_buf,
                                             uint32_t idesc)
{
    const uint64_t a0 = sdesc_sw128(a_buf, 16, 1024), b0 = sdesc_sw128(b_buf, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ao = ((kk >> 2) * (kOwn * 128) + (kk & 3) * 32) >> 4;
        const uint64_t bo = ((kk >> 2) * (STEP * 128) + (kk & 3) * 32) >> 4;
        if (kk == 0)
            mma_ss_w<0>(d_tmem, a0 + ao, b0 + bo, idesc);
        else
            mma_ss_w<1>(d_tmem, a0 + ao, b0 + bo, idesc);
    }
}

// D += A B over K = STEP streamed rows: A (128 x STEP, bf16 pairs) in TMEM at
// a_tmem, written by the math warps in chunks of 32 columns (chunk c's 32
// values packed into the first 16 of its own 32 columns); B the STEP-row tile
// in shared memory from column block b_buf on, MN-major.
template <int STEP>
__device__ __forceinline__ void issue_accumulate(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_buf,
                                                 uint32_t idesc, bool first)
{
    const uint64_t b0 = sdesc_sw128(b_buf, STEP * 128, 1024);
#pragma unroll
    for (int kk = 0; kk < STEP / 16; ++kk) {
        const uint32_t a = a_tmem + 32 * (kk >> 1) + 8 * (kk & 1);
        const uint64_t bo = (kk * 16 * 128) >> 4;
        if (kk == 0 && first)
            mma_ts_w<0>(d_tmem, a, b0 + bo, idesc);
        else
            mma_ts_w<1>(d_tmem, a, b0 + bo, idesc);
    }
}

// NC consecutive TMEM columns of this warp's lanes into r (warp-collective),
// and NC / 2 packed columns back.
template <int NC>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&r)[NC])
{
    if constexpr (NC == 32)
        tmem_ld32(taddr, r);
    else
        tmem_ld16(taddr, r);
}

template <int NC>
__device__ __forceinline__ void wait_cols(uint32_t (&r)[NC], uint32_t (&q)[NC])
{
    if constexpr (NC == 32) {
        tmem_wait_ld_r(r);
        tmem_bind_r(q);
    } else {
        tmem_wait_ld_r16(r);
        asm volatile(""
                     : "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]), "+r"(q[4]), "+r"(q[5]),
                       "+r"(q[6]), "+r"(q[7]), "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]),
                       "+r"(q[12]), "+r"(q[13]), "+r"(q[14]), "+r"(q[15])
                     :
                     : "memory");
    }
}

template <int NP>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&r)[NP])
{
    if constexpr (NP == 16) {
        tmem_st16(taddr, r);
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], "
                     "{%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                     "r"(r[6]), "r"(r[7])
                     : "memory");
    }
}

// 32 accumulator columns of this warp's 32 rows (fp32 in TMEM at taddr; the
// thread's lane is its row) * f -> bf16 at dst0 (the warp's first row, the
// chunk's first column; rows row_stride elements apart).  The values pass
// through the warp's 2 KB stage (row segments swizzled by row, so the writes
// are conflict-free) so that every global store instruction writes eight
// whole 64-byte row segments; rows n_valid and later are not written.
__device__ __forceinline__ void store_tile32(uint32_t taddr, float f, uint32_t stage, int lane,
                                             __nv_bfloat16 *dst0, size_t row_stride, int n_valid)
{
    uint32_t rr[32];
    tmem_ld32(taddr, rr);
    tmem_wait_ld_r(rr);
    const uint32_t row = stage + lane * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(row + ((c ^ ((lane >> 1) & 3)) << 4),
                     pack_bf16x2(__uint_as_float(rr[8 * c + 0]) * f, __uint_as_float(rr[8 * c + 1]) * f),
                     pack_bf16x2(__uint_as_float(rr[8 * c + 2]) * f, __uint_as_float(rr[8 * c + 3]) * f),
                     pack_bf16x2(__uint_as_float(rr[8 * c + 4]) * f, __uint_as_float(rr[8 * c + 5]) * f),
                     pack_bf16x2(__uint_as_float(rr[8 * c + 6]) * f, __uint_as_float(rr[8 * c + 7]) * f));
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rw = 8 * k + (lane >> 2), ch = lane & 3;
        const uint4 v = ld_shared_v4(stage + rw * 64 + ((ch ^ ((rw >> 1) & 3)) << 4));
        if (rw < n_valid)
            *reinterpret_cast<uint4 *>(dst0 + rw * row_stride + ch * 8) = v;
    }
    __syncwarp();
}

// ------------------------------------------------------------ the two main kernels

// One unit of work, decoded by the loading warp and handed to the others
// through a two-slot shared-memory ring.  dK/dV kernel: (kv head, 128-key
// tile, column half); dQ kernel: (head, 128-query tile).
struct BwdUnit {
    int b, t, head, dh;          // sequence, tile in it, (kv) head, column half
    int q0, lq, k0, lk;          // the sequence's rows and lengths
    int first, n_blk, n_steps;   // streamed blocks [first, first + n_blk); steps (x group)
    int valid;                   // 0: no more units
};

// Unit u of the dK/dV kernel (DQ false) or the dQ kernel (DQ true); `tiles`
// is the number of 128-row tiles of all sequences.
template <int D, bool DQ>
__device__ BwdUnit decode_unit(const BwdArgs &a, int u, int tiles)
{
    using C = BwdCfg<D, DQ>;
    constexpr int STEP = C::STEP;
    constexpr int SPLIT = DQ ? 1 : C::DSPLIT;
    BwdUnit w;
    const int per_head = tiles * SPLIT;
    const int n_heads = DQ ? a.num_heads : a.num_kv_heads;
    w.valid = u < per_head * n_heads;
    if (!w.valid)
        return w;
    w.head = u / per_head;
    const int r = u % per_head;
    // dQ: each head's tiles run last-first (a causal sequence's longest key
    // ranges first); dK/dV: in order (a sequence's first key tiles see the
    // most queries); a key tile's column halves are neighbours
    int gt = r / SPLIT;
    w.dh = r % SPLIT;
    if (DQ)
        gt = tiles - 1 - gt;
    const int32_t *start = DQ ? a.qtile_start : a.ktile_start;
    w.b = owner_of(start, a.batch, gt);
    w.t = gt - start[w.b];
    w.q0 = a.cu_q[w.b];
    w.lq = a.cu_q[w.b + 1] - w.q0;
    w.k0 = a.cu_k[w.b];
    w.lk = a.cu_k[w.b + 1] - w.k0;
    const long long off = a.causal == 2 ? w.lk - w.lq : 0;
    const int wl = a.window_left;
    long long lo, hi;
    if (!DQ) {
        // queries that see a key of this tile: i >= j - off (causal),
        // i <= j - off + window_left (window)
        const int j_lo = w.t * kOwn, j_hi = min(w.lk, j_lo + kOwn);
        lo = a.causal ? max(0ll, j_lo - off) : 0;
        hi = w.lq - 1;
        if (wl >= 0)
            hi = min(hi, static_cast<long long>(j_hi) - 1 - off + wl);
    } else {
        // keys some row of this tile sees: j <= i + off (causal), j >= i + off
        // - window_left (window)
        const int i_lo = w.t * kOwn, i_hi = min(w.lq, i_lo + kOwn);
        lo = (a.causal && wl >= 0) ? max(0ll, i_lo + off - wl) : 0;
        hi = w.lk - 1;
        if (a.causal)
            hi = min(hi, static_cast<long long>(i_hi) - 1 + off);
    }
    w.first = lo <= hi ? static_cast<int>(lo / STEP) : 0;
    w.n_blk = lo <= hi ? static_cast<int>(hi / STEP) + 1 - w.first : 0;
    w.n_steps = DQ ? w.n_blk : w.n_blk * (a.num_heads / a.num_kv_heads);
    return w;
}

// Persistent CTAs, one per SM, take units from an atomic counter.  Warp 0
// loads (the unit's own 128-row tiles once, the streamed tiles per step),
// warp 1 issues the MMAs, warps 4-11 do the elementwise work: warp w owns
// TMEM lanes (own rows) 32 (w % 4) .. +31; warpgroup g = (w - 4) / 4 takes
// the steps held in TMEM buffer g, all STEP columns of each.
//
// dK/dV kernel (DQ false): own = K, V of a key tile; a step is a block of
// STEP queries of one query head of the group; per step
//   MMA:  S^T = K Q^T, dP^T = V dO^T -> buffer x (s_full(x));
//         then, for the previous step: dV += P^T dO, dK += dS^T Q
//   math: P^T = 2^(s scale log2e - lse log2e) (masked: 0), dS^T = P^T (dP^T -
//         Delta) -> bf16 over S^T / dP^T (p_full(x))
// dQ kernel (DQ true): own = Q, dO of a query tile; a step is a block of
// STEP keys; S = Q K^T, dP = dO V^T; dS (over dP); dQ += dS K.
//
// Across units nothing restarts: the step counter (ring stage, TMEM buffer
// and their barrier phases) runs on, the next unit's own tiles load as soon
// as the last score products of the current one have read the old ones, and
// the next unit's first scores run during the current unit's epilogue; only
// its first accumulating product waits for the epilogue (epi_done) to have
// read the accumulators.
template <int D, bool DQ>
__global__ void __launch_bounds__(kThreads, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a)
{
    using C = BwdCfg<D, DQ>;
    constexpr int DB = C::DB, NSTAGE = C::NSTAGE, STEP = C::STEP, NCH = C::NCH;
    constexpr int NACC = DQ ? D : C::DKV;        // accumulator columns (each)
    constexpr int DH = NACC / 2;                  // accumulator columns per math thread
    constexpr uint32_t BUF = DQ ? C::Q_BUF : C::KV_BUF;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ BwdUnit s_unit[2];

    // The dQ kernel, launched next with programmatic dependent launch, reads
    // nothing this kernel writes: let it take each SM this kernel's CTAs leave.
    if (!DQ)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*a.status != VFA_OK)
        return;
    const int B = a.batch, H = a.num_heads, Hkv = a.num_kv_heads;
    const int tiles = DQ ? a.qtile_start[B] : a.ktile_start[B];
    int32_t *counter = a.status + (DQ ? 2 : 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int half = warp >= kFirstMathWarp ? (warp - kFirstMathWarp) >> 2 : 0;
    const int r = quarter * 32 + lane;            // own row of math threads

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sOwn0 = base, sOwn1 = sOwn0 + C::OWN_BYTES;     // K, V  /  Q, dO
    const uint32_t sRing = sOwn1 + C::OWN_BYTES;                    // stage: Q, dO  /  K, V
    const uint32_t sStat = sRing + NSTAGE * C::STAGE_BYTES;         // per math warp: nl, -Delta
    const uint32_t sEpi = sStat + kMathWarps * C::STAT_BYTES;       // per math warp: output stage
    const uint32_t bars = sEpi + kMathWarps * kEpiStage;
    auto ring_full = [&](int st) { return bars + 8u * st; };
    auto ring_empty = [&](int st) { return bars + 8u * (NSTAGE + st); };
    auto s_full = [&](int x) { return bars + 8u * (2 * NSTAGE + x); };
    auto p_full = [&](int x) { return bars + 8u * (2 * NSTAGE + 2 + x); };
    auto unit_full = [&](int x) { return bars + 8u * (2 * NSTAGE + 4 + x); };
    auto unit_empty = [&](int x) { return bars + 8u * (2 * NSTAGE + 6 + x); };
    const uint32_t own_full = bars + 8u * (2 * NSTAGE + 8);
    const uint32_t own_empty = bars + 8u * (2 * NSTAGE + 9);
    const uint32_t acc_done = bars + 8u * (2 * NSTAGE + 10);
    const uint32_t epi_done = bars + 8u * (2 * NSTAGE + 11);
    const uint32_t drain_bar = bars + 8u * (2 * NSTAGE + 12);
    auto stage0 = [&](int st) { return sRing + st * C::STAGE_BYTES; };
    auto stage1 = [&](int st) { return sRing + st * C::STAGE_BYTES + C::STEP_BYTES; };
    volatile int *abort = &s_abort;

    if (tid == 0) {
        s_abort = 0;
        for (int st = 0; st < NSTAGE; ++st) {
            mbar_init(ring_full(st), 1);
            mbar_init(ring_empty(st), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), kMathThreads / 2);    // buffer x's warpgroup
            mbar_init(unit_full(x), 1);
            mbar_init(unit_empty(x), 1 + kMathWarps);
        }
        mbar_init(own_full, 1);
        mbar_init(own_empty, 1);
        mbar_init(acc_done, 1);
        mbar_init(epi_done, kMathThreads);
        mbar_init(drain_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    // Consumers take unit n from the ring; false at the end (or on abort).
    auto take_unit = [&](uint32_t n, BwdUnit &w) -> bool {
        if (!mbar_wait_warp(unit_full(n & 1), (n >> 1) & 1u, abort))
            return false;
        w = s_unit[n & 1];
        return w.valid;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            tma_prefetch_map(&a.tm_q);
            tma_prefetch_map(&a.tm_k);
            tma_prefetch_map(&a.tm_v);
            tma_prefetch_map(&a.tm_do);
            const CUtensorMap *own0 = DQ ? &a.tm_q : &a.tm_k, *own1 = DQ ? &a.tm_do : &a.tm_v;
            const CUtensorMap *str0 = DQ ? &a.tm_ks : &a.tm_qs, *str1 = DQ ? &a.tm_vs : &a.tm_dos;
            tma_prefetch_map(str0);
            tma_prefetch_map(str1);
            uint32_t g = 0, owns = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                if (!mbar_wait(unit_empty(n & 1), ((n >> 1) & 1u) ^ 1u, abort))
                    break;
                const BwdUnit w = decode_unit<D, DQ>(a, atomicAdd(counter, 1), tiles);
                s_unit[n & 1] = w;
                mbar_arrive(unit_full(n & 1));
                if (!w.valid)
                    break;
                if (w.n_steps == 0)
                    continue;
                // the previous unit's score products have read the own tiles
                if (!mbar_wait(own_empty, (owns & 1u) ^ 1u, abort))
                    break;
                mbar_arrive_expect_tx(own_full, 2 * C::OWN_BYTES);
                const int own_row = (DQ ? w.q0 : w.k0) + w.t * kOwn;
                load_rows<DB, C::OWN_BOX>(sOwn0, own0, own_full, w.head, own_row, kOwn);
                load_rows<DB, C::OWN_BOX>(sOwn1, own1, own_full, w.head, own_row, kOwn);
                ++owns;
                const int group = H / Hkv;
                for (int s = 0; s < w.n_steps; ++s, ++g) {
                    const int st = g % NSTAGE;
                    if (!mbar_wait(ring_empty(st), ((g / NSTAGE) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(ring_full(st), C::STAGE_BYTES);
                    // dK/dV: step s = (query head of the group, query block);
                    // dQ: key block of the head's kv head
                    const int blk = w.first + (DQ ? s : s % w.n_blk);
                    const int row = (DQ ? w.k0 : w.q0) + blk * STEP;
                    const int head = DQ ? w.head / group : w.head * group + s / w.n_blk;
                    load_rows<DB, STEP>(stage0(st), str0, ring_full(st), head, row, STEP);
                    load_rows<DB, STEP>(stage1(st), str1, ring_full(st), head, row, STEP);
                }
            }
            if (*abort) {
                // the last fill of each stage and of the own tiles may be in flight
                if (owns > 0)
                    mbar_wait_drain(own_full, (owns - 1) & 1u);
                for (int st = 0; st < NSTAGE; ++st) {
                    const uint32_t fills = g / NSTAGE + (static_cast<uint32_t>(st) < g % NSTAGE ? 1u : 0u);
                    if (fills > 0)
                        mbar_wait_drain(ring_full(st), (fills - 1) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // All 32 lanes run this loop on warp-uniform values; one elected lane
        // issues each MMA and commit.
        uint32_t g = 0, owns = 0, units = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            BwdUnit w;
            const bool more = take_unit(n, w);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(unit_empty(n & 1));
            if (!more)
                break;
            if (w.n_steps == 0)
                continue;
            if (!mbar_wait_warp(own_full, owns & 1u, abort)) {
                ok = false;
                break;
            }
            ++owns;
            // this unit's column half of the streamed tiles' columns (dK/dV at
            // head_dim 256): DKV / 64 column blocks on
            const uint32_t col0 = DQ ? 0u : w.dh * (C::DKV / 64) * (STEP * 128);
            for (int s = 0; s <= w.n_steps && ok; ++s) {
                if (s < w.n_steps) {
                    const uint32_t gs = g + s;
                    const int st = gs % NSTAGE, x = gs & 1;
                    if (!mbar_wait_warp(ring_full(st), (gs / NSTAGE) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // buffer x was last read by step gs - 2's products, issued earlier
                    const uint32_t buf = tmem + BUF + C::BUF_STRIDE * x;
                    issue_scores<D, STEP>(buf, sOwn0, stage0(st), C::IDESC_T);
                    issue_scores<D, STEP>(buf + STEP, sOwn1, stage1(st), C::IDESC_T);
                    mma_commit_w(s_full(x));
                    if (s == w.n_steps - 1)
                        mma_commit_w(own_empty);        // own tiles free once these complete
                }
                if (s >= 1) {
                    const uint32_t gp = g + s - 1;
                    const int stp = gp % NSTAGE, xp = gp & 1;
                    if (!mbar_wait_warp(p_full(xp), (gp >> 1) & 1u, abort) ||
                        (s == 1 && !mbar_wait_warp(epi_done, (units & 1u) ^ 1u, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t buf = tmem + BUF + C::BUF_STRIDE * xp;
                    if (DQ) {
                        issue_accumulate<STEP>(tmem + C::COL_DQ, buf + STEP, stage0(stp),
                                               C::IDESC_DQ, s == 1);
                    } else {
                        issue_accumulate<STEP>(tmem + C::COL_DV, buf, stage1(stp) + col0,
                                               C::IDESC_KV, s == 1);
                        issue_accumulate<STEP>(tmem + C::COL_DK, buf + STEP, stage0(stp) + col0,
                                               C::IDESC_KV, s == 1);
                    }
                    mma_commit_w(ring_empty(stp));
                }
            }
            if (!ok)
                break;
            mma_commit_w(acc_done);
            g += w.n_steps;
            ++units;
        }
        if (!ok || *abort) {
            mma_commit_w(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else if (warp >= kFirstMathWarp) {
        // ------------------------------------------------------------ elementwise, epilogue
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        // per warp and 32-column chunk: 32 nl, then 32 -Delta
        const uint32_t wstat = sStat + (warp - kFirstMathWarp) * C::STAT_BYTES;
        float *stat = reinterpret_cast<float *>(smem_raw + (wstat - raw));
        const float scale_log2 = a.scale_log2;
        uint32_t g = 0, units = 0;
        bool ok = true;
        __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(a.dq);
        __nv_bfloat16 *dk = static_cast<__nv_bfloat16 *>(a.dk);
        __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(a.dv);
        for (uint32_t n = 0; ok; ++n) {
            BwdUnit w;
            const bool more = take_unit(n, w);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(unit_empty(n & 1));
            if (!more)
                break;
            const long long off = a.causal == 2 ? w.lk - w.lq : 0;
            const int wl = a.window_left;
            const int own = w.t * kOwn + r;       // this thread's own row (key or query)
            // where this thread's accumulator columns go
            size_t row_out;
            if (DQ)
                row_out = (static_cast<size_t>(w.q0 + own) * H + w.head) * D + half * DH;
            else
                row_out = (static_cast<size_t>(w.k0 + own) * Hkv + w.head) * D + w.dh * C::DKV +
                          half * DH;
            const bool own_valid = DQ ? own < w.lq : own < w.lk;
            if (w.n_steps == 0) {
                // no key / query pairs: zero gradients
                if (own_valid) {
#pragma unroll
                    for (int d = 0; d < DH; d += 8) {
                        if (DQ) {
                            *reinterpret_cast<uint4 *>(dq + row_out + d) = make_uint4(0, 0, 0, 0);
                        } else {
                            *reinterpret_cast<uint4 *>(dk + row_out + d) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(dv + row_out + d) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                continue;
            }
            // dQ: this thread's row constants
            float nl_row = 0.f, nd_row = 0.f;
            if (DQ && own_valid) {
                const size_t srow = static_cast<size_t>(w.q0 + own) * H + w.head;
                nl_row = -a.lse[srow] * kLog2e;
                nd_row = -a.delta[srow];
            }
            const int group = H / Hkv;
            // The two warpgroups take the steps in turn (warpgroup x the steps
            // in TMEM buffer x), each doing all STEP columns of its rows in
            // chunks of 32, so two steps are in the works at once.
            for (int s = (half - static_cast<int>(g & 1u)) & 1; s < w.n_steps && ok; s += 2) {
                const uint32_t gs = g + s;
                const int x = gs & 1;
                const int blk = w.first + (DQ ? s : s % w.n_blk);
                const int c0 = blk * STEP;                 // the step's first streamed column
                if (!DQ) {
                    // -lse log2(e) and -Delta of the step's query columns
                    const int hq = w.head * group + s / w.n_blk;
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const int i = c0 + 32 * c + lane;
                        const size_t srow = static_cast<size_t>(w.q0 + i) * H + hq;
                        stat[64 * c + lane] = i < w.lq ? -a.lse[srow] * kLog2e : 0.f;
                        stat[64 * c + 32 + lane] = i < w.lq ? -a.delta[srow] : 0.f;
                    }
                    __syncwarp();
                }
                // a step every (own, streamed) pair of which is visible needs no mask
                const long long slo = static_cast<long long>(c0);
                const long long olo = static_cast<long long>(w.t) * kOwn;
                bool full;
                if (DQ)
                    full = slo + STEP <= w.lk && olo + kOwn <= w.lq &&
                           (!a.causal || slo + STEP - 1 <= olo + off) &&
                           (wl < 0 || slo >= olo + kOwn - 1 + off - wl);
                else
                    full = olo + kOwn <= w.lk && slo + STEP <= w.lq &&
                           (!a.causal || olo + kOwn - 1 <= slo + off) &&
                           (wl < 0 || olo >= slo + STEP - 1 + off - wl);
                ok = mbar_wait_warp(s_full(x), (gs >> 1) & 1u, abort);
                if (!ok)
                    break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    const uint32_t st_addr = tmem + lane_addr + BUF + C::BUF_STRIDE * x + 32 * c;
                    uint32_t sr[32], dr[32];
                    ld_cols<32>(st_addr, sr);
                    ld_cols<32>(st_addr + STEP, dr);
                    wait_cols<32>(sr, dr);
                    uint32_t dk2[16];
                    const int cb = c0 + 32 * c;            // the chunk's first streamed column
                    if (DQ) {
                        if (full) {
                            query_row_grads<false, 32>(sr, dr, scale_log2, nl_row, nd_row, 0, 32,
                                                       dk2);
                        } else {
                            int lo, hi;
                            query_row_span(own, cb, w.lk, w.lq, a.causal, wl, off, &lo, &hi);
                            query_row_grads<true, 32>(sr, dr, scale_log2, nl_row, nd_row, lo, hi,
                                                      dk2);
                        }
                    } else {
                        uint32_t pk[16];
                        const uint32_t cstat = wstat + 256 * c;
                        if (full) {
                            key_row_grads<false, 32>(sr, dr, scale_log2, cstat, 0, 32, pk, dk2);
                        } else {
                            int lo, hi;
                            key_row_span(own, cb, w.lk, w.lq, a.causal, wl, off, &lo, &hi);
                            key_row_grads<true, 32>(sr, dr, scale_log2, cstat, lo, hi, pk, dk2);
                        }
                        // P^T (bf16 pairs) over the first half of the chunk's S^T columns
                        st_cols<16>(st_addr, pk);
                    }
                    // dS (bf16 pairs) over the first half of the chunk's dP columns
                    st_cols<16>(st_addr + STEP, dk2);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full(x));
            }
            if (!ok)
                break;
            ok = mbar_wait_warp(acc_done, units & 1u, abort);
            if (!ok)
                break;
            tc_fence_after();
            {
                // this warp's 32 rows start at own row w.t * 128 + 32 * quarter
                const int wrow = w.t * kOwn + quarter * 32;
                const int n_valid = (DQ ? w.lq : w.lk) - wrow;
                const uint32_t stage = sEpi + (warp - kFirstMathWarp) * kEpiStage;
                const size_t stride = static_cast<size_t>(DQ ? H : Hkv) * D;
                const size_t base_out = row_out - static_cast<size_t>(lane) * stride;
#pragma unroll 1
                for (int cb = 0; cb < DH; cb += 32) {
                    if (DQ) {
                        store_tile32(tmem + lane_addr + C::COL_DQ + half * DH + cb, a.scale, stage,
                                     lane, dq + base_out + cb, stride, n_valid);
                    } else {
                        store_tile32(tmem + lane_addr + C::COL_DV + half * DH + cb, 1.f, stage,
                                     lane, dv + base_out + cb, stride, n_valid);
                        store_tile32(tmem + lane_addr + C::COL_DK + half * DH + cb, a.scale, stage,
                                     lane, dk + base_out + cb, stride, n_valid);
                    }
                }
            }
            // the accumulators may be overwritten by the next unit's products
            tc_fence_before();
            mbar_arrive(epi_done);
            g += w.n_steps;
            ++units;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort && tid == 0)
        atomicCAS(a.status, VFA_OK, VFA_ERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs &a, int key_tile_bound, int q_tile_bound, int sm_count,
                         cudaStream_t s)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !attr_done[dev]) {
        if ((e = cudaFuncSetAttribute(bwd_main_kernel<D, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(BwdCfg<D, false>::SMEM))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(bwd_main_kernel<D, true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(BwdCfg<D, true>::SMEM))) != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    bwd_prep_kernel<<<1, kPrepThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    bwd_delta_kernel<D><<<sm_count * 8, 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    // persistent grids: one CTA per SM (fewer when there are fewer units)
    const long long kv_units =
        static_cast<long long>(key_tile_bound) * BwdCfg<D, false>::DSPLIT * a.num_kv_heads;
    const long long q_units = static_cast<long long>(q_tile_bound) * a.num_heads;
    if (kv_units > 0) {
        bwd_main_kernel<D, false><<<static_cast<int>(std::min<long long>(kv_units, sm_count)),
                                    kThreads, BwdCfg<D, false>::SMEM, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    if (q_units > 0) {
        // Programmatic dependent launch: the dQ kernel's CTAs start on the SMs
        // the dK/dV kernel's CTAs leave, without waiting for the whole grid.  It
        // reads only the prep and Delta kernels' output, complete before the
        // dK/dV kernel started (a plain launch after them), so it needs no
        // griddepcontrol.wait; its atomic unit counter balances CTAs that start
        // late.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(std::min<long long>(q_units, sm_count)));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = BwdCfg<D, true>::SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = kv_units > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, bwd_main_kernel<D, true>, a)) != cudaSuccess)
            return e;
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace

size_t bwd_workspace_bytes(int batch, int total_q, int num_heads, int head_dim)
{
    (void)head_dim;
    size_t n = 256;                                                   // status word
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);          // key tile starts
    n = (n + 255) & ~static_cast<size_t>(255);
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);          // q tile starts
    n = (n + 255) & ~static_cast<size_t>(255);
    n += static_cast<size_t>(total_q) * num_heads * sizeof(float);    // Delta
    return (n + 255) & ~static_cast<size_t>(255);
}

void bwd_workspace_split(void *ws, int batch, int total_q, int num_heads, BwdArgs *a)
{
    (void)total_q;
    (void)num_heads;
    uint8_t *p = static_cast<uint8_t *>(ws);
    a->status = reinterpret_cast<int32_t *>(p);
    size_t n = 256;
    a->ktile_start = reinterpret_cast<int32_t *>(p + n);
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);
    n = (n + 255) & ~static_cast<size_t>(255);
    a->qtile_start = reinterpret_cast<int32_t *>(p + n);
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);
    n = (n + 255) & ~static_cast<size_t>(255);
    a->delta = reinterpret_cast<float *>(p + n);
}

cudaError_t launch_bwd(int head_dim, const BwdArgs &a, int key_tile_bound, int q_tile_bound,
                       int sm_count, cudaStream_t stream)
{
    switch (head_dim) {
    case 64: return launch_bwd_d<64>(a, key_tile_bound, q_tile_bound, sm_count, stream);
    case 128: return launch_bwd_d<128>(a, key_tile_bound, q_tile_bound, sm_count, stream);
    case 256: return launch_bwd_d<256>(a, key_tile_bound, q_tile_bound, sm_count, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vfa
