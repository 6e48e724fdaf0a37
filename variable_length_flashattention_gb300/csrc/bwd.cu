// bwd.cu -- variable-length attention backward on sm_103a (head_dim 64, 128).
//
// Gradients of the forward (scaled scores, causal / bottom-right / sliding-
// window masks on local positions, softmax over the visible keys) for an
// upstream gradient dO, given the forward's out and natural-log lse.  With
// P = exp(scale * q.k - lse), dP = dO V^T, Delta = rowsum(dO * out) and
// dS = P * (dP - Delta):
//   dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K.
//
// Four kernels:
//   * bwd_prep: one CTA validates cu_seqlens and writes each sequence's first
//     global key tile (a prefix sum of ceil(Lk_b / 128));
//   * bwd_delta: Delta[t, h] = sum_d dO * out, one warp per (token, head);
//   * bwd_kernel: one CTA per (128-key tile, kv head).  K and V stay in
//     shared memory; for every query head of the group and every 128-row q
//     tile that sees one of the tile's keys, TMA brings Q and dO (two
//     buffers, so the next tile's copies overlap this one's work), and
//     tcgen05.mma computes S^T = K Q^T and dP^T = V dO^T into TMEM, one
//     64-query half at a time; for each half in turn, two threads per key
//     row form P^T (bf16, back into TMEM over the S^T columns) and dS^T (bf16,
//     128-byte-swizzled shared memory), and more MMAs accumulate dV += P^T dO
//     and dK += dS^T Q in TMEM across the whole loop; after both halves,
//     dQ = dS K for this q tile, which the threads (now two per query row)
//     add into an fp32 buffer with vector atomics.  At the end dK (scaled) and
//     dV leave as bf16;
//   * bwd_dq: dQ = bf16(scale * the fp32 sum).
// TMEM: S^T 128 columns, dP^T 128 (dQ reuses them once dP is read), dV and
// dK D each -- 512 for D = 128.  Every wait is bounded; on expiry the CTA
// records VFA_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cfloat>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

constexpr int kT = 128;            // key rows and query rows per tile
constexpr int kComputeWarps = 8;   // two threads per tile row
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;   // + the TMA / MMA issuing warp
constexpr int kPrepThreads = 1024;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int DB = D / 64;                       // 64-column blocks per row
    static constexpr uint32_t TILE_BYTES = kT * D * 2;      // a 128-row tile of K, V, Q or dO
    static constexpr uint32_t PS_BYTES = kT * kT * 2;       // dS^T, 128 x 128 bf16
    static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 256 + D;
    static constexpr uint32_t COL_DQ = COL_DPT;             // dQ takes dP^T's columns
    // P^T (bf16 pairs) goes over the S^T columns: queries 0-63 to columns
    // 0-31, queries 64-127 to columns 64-95
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NUM_BARS = 11;
    // K, V, two Q and two dO buffers, dS^T, lse, Delta, barriers
    static constexpr size_t SMEM = 1024 + 6 * TILE_BYTES + PS_BYTES + 2 * kT * 4 +
                                   NUM_BARS * 8 + 64;
    static constexpr uint32_t IDESC_T = idesc_bf16_f32(kT, 64, false, false);   // S^T, dP^T halves
    static constexpr uint32_t IDESC_KV = idesc_bf16_f32(kT, D, false, true);    // dV, dK
    static constexpr uint32_t IDESC_Q = idesc_bf16_f32(kT, D, true, true);      // dQ
    static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// ------------------------------------------------------------ prep

__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const BwdArgs a)
{
    __shared__ int warp_sums[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.batch;
    if (tid == 0)
        s_bad = (a.cu_q[0] != 0 || a.cu_k[0] != 0 || a.cu_q[B] != a.total_q ||
                 a.cu_k[B] != a.total_k);
    __syncthreads();
    int carry = 0;
    for (int base = 0; base < B; base += kPrepThreads) {
        const int b = base + tid;
        int nt = 0;
        if (b < B) {
            const int lq = a.cu_q[b + 1] - a.cu_q[b], lk = a.cu_k[b + 1] - a.cu_k[b];
            if (lq < 0 || lk < 0)
                s_bad = 1;
            else
                nt = (lk + kT - 1) / kT;
        }
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
            a.ktile_start[b] = carry + excl;
        carry += warp_sums[31];
        __syncthreads();
    }
    if (tid == 0) {
        a.ktile_start[B] = carry;
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

// ------------------------------------------------------------ main

// Byte offset of the 16-byte chunk holding columns 8*c8 .. 8*c8+7 of row r in
// a 128-row operand of 128 bf16 columns stored as two 64-column blocks with
// the 128-byte swizzle (the layout TMA's SWIZZLE_128B gives).
__device__ __forceinline__ uint32_t sw_chunk(int r, int c8)
{
    return static_cast<uint32_t>((c8 >> 3) * (kT * 128) + r * 128 + (((c8 & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr)
{
    const uint4 v = ld_shared_v4(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

// Where the key row of this thread sees query column c of the tile (only
// for tiles that are not fully visible).
struct BwdMask {
    int j, lk, lq, causal, wl;
    long long i_lo, off;
    __device__ __forceinline__ bool visible(int c) const
    {
        const long long i = i_lo + c;
        bool v = j < lk && i < lq;
        if (causal)
            v = v && j <= i + off;
        if (wl >= 0)
            v = v && j >= i + off - wl;
        return v;
    }
};

// P^T and dS^T of one 16-column chunk of this thread's key row: p = 2^(s *
// scale_log2 - lse2) (masked entries 0), ds = p * (dp - Delta); lse2 and
// Delta of the chunk's columns come from shared memory (nl = -lse2).  The
// bf16 pairs land in pk[0..7] and dk2[0..7].
template <bool FULL>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&sr)[16], const uint32_t (&dr)[16],
                                          float scale_log2, uint32_t s_nl, uint32_t s_delta,
                                          int cb, const BwdMask &m, uint32_t *pk, uint32_t *dk2)
{
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        const float4 nl = ld_shared_f4(s_nl + (cb + e) * 4);
        const float4 dl = ld_shared_f4(s_delta + (cb + e) * 4);
        const float nls[4] = {nl.x, nl.y, nl.z, nl.w};
        const float dls[4] = {dl.x, dl.y, dl.z, dl.w};
        float p[4], d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float x = ex2_approx(fmaf(__uint_as_float(sr[e + u]), scale_log2, nls[u]));
            p[u] = FULL ? x : (m.visible(cb + e + u) ? x : 0.f);
            d[u] = p[u] * (__uint_as_float(dr[e + u]) - dls[u]);
        }
        pk[(e >> 1)] = pack_bf16x2(p[0], p[1]);
        pk[(e >> 1) + 1] = pack_bf16x2(p[2], p[3]);
        dk2[(e >> 1)] = pack_bf16x2(d[0], d[1]);
        dk2[(e >> 1) + 1] = pack_bf16x2(d[2], d[3]);
    }
}

// Adds this thread's dQ row segment (DH floats) into the fp32 sum.
template <int DH>
__device__ __forceinline__ void flush_dq(float4 *dst, const float4 (&acc)[DH / 4])
{
#pragma unroll
    for (int c = 0; c < DH / 4; ++c)
        atomicAdd(dst + c, acc[c]);
}

// Warps 0-7 compute (warp w: TMEM lanes / tile rows 32 (w % 4) .. +31; of
// each 64-query half the 32 queries 32 (w / 4) .. +31; of dQ, dK and dV the
// column half w / 4); warp 8 issues the TMA copies and the MMAs.
//
// Per step s (one query head, one q tile):
//   issuer:  per query half h (64 columns): S^T_h, dP^T_h -> bar_s<h> (S^T_0
//            right away, dP^T once step s-1's dQ, which it overwrites, has
//            been read; that also frees step s-1's Q / dO buffer for step
//            s+1's copies); [P^T_h in TMEM, dS^T_h in shared memory, bar_p<h>]
//            dV += P^T_h dO_h (A from TMEM), dK += dS^T_h Q_h; after half 1,
//            dQ = dS K -> bar_m2;
//   compute: lse, Delta -> shared (bar_ld); for h = 0, 1 in turn, all eight
//            warps: [bar_s<h>] P^T = exp(S^T scale - lse) into TMEM over the
//            S^T columns it has read, dS^T = P^T (dP^T - Delta) into shared
//            memory (bar_p<h>); the previous step's dQ rows
//            into the fp32 sum with vector atomics while the tensor core runs
//            this step's products; [bar_m2] this step's dQ rows out of TMEM
//            into registers (bar_dq).
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_kernel(const __grid_constant__ BwdArgs a)
{
    using C = BwdCfg<D>;
    constexpr int DB = C::DB;
    constexpr int DH = D / 2;                     // columns of dQ, dK, dV per thread
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

    if (*a.status != VFA_OK)
        return;
    const int B = a.batch, H = a.num_heads, Hkv = a.num_kv_heads;
    const int gt = blockIdx.x, kh = blockIdx.y;
    if (gt >= a.ktile_start[B])
        return;
    int lo = 0, hi = B - 1;                       // largest b with ktile_start[b] <= gt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.ktile_start[mid] <= gt)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int b = lo, kt = gt - a.ktile_start[b];
    const int q0 = a.cu_q[b], lq = a.cu_q[b + 1] - q0;
    const int k0 = a.cu_k[b], lk = a.cu_k[b + 1] - k0;
    const long long off = a.causal == 2 ? lk - lq : 0;
    const int wl = a.window_left;
    const int j_lo = kt * kT, j_hi = min(lk, j_lo + kT);
    // query rows that see a key of this tile: i >= j - off (causal) and
    // i <= j - off + window_left (window)
    long long i_min = a.causal ? max(0ll, j_lo - off) : 0;
    long long i_max = lq - 1;
    if (wl >= 0)
        i_max = min(i_max, static_cast<long long>(j_hi) - 1 - off + wl);
    const int it0 = i_min <= i_max ? static_cast<int>(i_min / kT) : 0;
    const int n_it = i_min <= i_max ? static_cast<int>(i_max / kT) + 1 - it0 : 0;
    const int group = H / Hkv;
    const int n_steps = n_it * group;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = (warp & 3) * 32 + lane;         // tile row (TMEM lane) of compute threads
    const int half = (warp >> 2) & 1;             // column half of compute threads
    const int sub = half;                         // their 32-query slice within a query half
    const int j = j_lo + r;                       // key (local position) of row r
    __nv_bfloat16 *dk = static_cast<__nv_bfloat16 *>(a.dk);
    __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(a.dv);

    if (n_steps == 0) {
        // no query sees these keys: zero gradients
        if (warp < kComputeWarps && j < lk) {
            const size_t row = (static_cast<size_t>(k0 + j) * Hkv + kh) * D + half * DH;
#pragma unroll
            for (int d = 0; d < DH; d += 8) {
                *reinterpret_cast<uint4 *>(dk + row + d) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dv + row + d) = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sK = base, sV = sK + C::TILE_BYTES;
    const uint32_t sQ = sV + C::TILE_BYTES;           // two buffers
    const uint32_t sDO = sQ + 2 * C::TILE_BYTES;      // two buffers
    const uint32_t sDS = sDO + 2 * C::TILE_BYTES;
    const uint32_t sLse = sDS + C::PS_BYTES, sDelta = sLse + kT * 4;
    const uint32_t bars = sDelta + kT * 4;
    const uint32_t bar_kv = bars, bar_s0 = bars + 8, bar_s1 = bars + 16, bar_m2 = bars + 24;
    const uint32_t bar_ld = bars + 32, bar_p0 = bars + 40, bar_p1 = bars + 48;
    const uint32_t bar_dq = bars + 56, bar_drain = bars + 64;
    auto bar_q = [&](int x) { return bars + 72 + 8u * x; };
    float *nl_s = reinterpret_cast<float *>(smem_raw + (sLse - raw));     // -lse * log2(e)
    float *delta_s = reinterpret_cast<float *>(smem_raw + (sDelta - raw));
    volatile int *abort = &s_abort;

    if (tid == 0) {
        s_abort = 0;
        mbar_init(bar_kv, 1);
        mbar_init(bar_q(0), 1);
        mbar_init(bar_q(1), 1);
        mbar_init(bar_s0, 1);
        mbar_init(bar_s1, 1);
        mbar_init(bar_m2, 1);
        mbar_init(bar_ld, kComputeThreads);
        mbar_init(bar_p0, kComputeThreads);
        mbar_init(bar_p1, kComputeThreads);
        mbar_init(bar_dq, kComputeThreads);
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    // step s -> (query head, q tile)
    auto step_hq = [&](int s) { return kh * group + s / n_it; };
    auto step_it = [&](int s) { return it0 + s % n_it; };

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ issuer
        // All 32 lanes run this loop on warp-uniform values; one elected lane
        // issues each MMA and commit, lane 0 the copies.
        if (lane == 0) {
            tma_prefetch_map(&a.tm_q);
            tma_prefetch_map(&a.tm_k);
            tma_prefetch_map(&a.tm_v);
            tma_prefetch_map(&a.tm_do);
        }
        auto load_q = [&](int s) {
            if (lane == 0) {
                const int x = s & 1;
                mbar_arrive_expect_tx(bar_q(x), 2 * C::TILE_BYTES);
                const int row = q0 + step_it(s) * kT, hq = step_hq(s);
                for (int db = 0; db < DB; ++db) {
                    tma_load_3d(sQ + x * C::TILE_BYTES + db * (kT * 128), &a.tm_q, bar_q(x),
                                db * 64, hq, row);
                    tma_load_3d(sDO + x * C::TILE_BYTES + db * (kT * 128), &a.tm_do, bar_q(x),
                                db * 64, hq, row);
                }
            }
            __syncwarp();
        };
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_kv, 2 * C::TILE_BYTES);
            for (int db = 0; db < DB; ++db) {
                tma_load_3d(sK + db * (kT * 128), &a.tm_k, bar_kv, db * 64, kh, k0 + j_lo);
                tma_load_3d(sV + db * (kT * 128), &a.tm_v, bar_kv, db * 64, kh, k0 + j_lo);
            }
        }
        load_q(0);
        int q_loads = 1;
        if (n_steps > 1) {
            load_q(1);
            q_loads = 2;
        }
        const uint64_t k_d = sdesc_sw128(sK, 16, 1024), v_d = sdesc_sw128(sV, 16, 1024);
        const uint64_t k_mn = sdesc_sw128(sK, kT * 128, 1024);
        const uint64_t ds_d = sdesc_sw128(sDS, 16, 1024);
        const uint64_t ds_mn = sdesc_sw128(sDS, kT * 128, 1024);
        // S^T_h or dP^T_h = (K or V) (Q or dO)^T for query half h (N = 64):
        // queries 64 h .. 64 h + 63 start 64 h rows into each 64-column block
        auto issue_t = [&](uint32_t d_col, uint64_t a_d, uint32_t b_buf, int h) {
            const uint64_t b_d = sdesc_sw128(b_buf + h * 64 * 128, 16, 1024);
            mma_ss_w<0>(tmem + d_col + h * 64, a_d, b_d, C::IDESC_T);
#pragma unroll
            for (int kk = 1; kk < D / 16; ++kk) {
                const uint32_t o16 = ((kk >> 2) * (kT * 128) + (kk & 3) * 32) >> 4;
                mma_ss_w<1>(tmem + d_col + h * 64, a_d + o16, b_d + o16, C::IDESC_T);
            }
        };
        // dV += P^T dO and dK += dS^T Q over the queries of half h (K = 64)
        auto issue_kv = [&](int h, uint32_t x, bool first) {
            const uint64_t do_mn = sdesc_sw128(sDO + x * C::TILE_BYTES, kT * 128, 1024);
            const uint64_t q_mn = sdesc_sw128(sQ + x * C::TILE_BYTES, kT * 128, 1024);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int kk = h * 4 + k4;
                // P^T of queries 16 kk .. +15: bf16 pairs at columns 64 h +
                // 32 (k4 / 2) + 8 (k4 % 2), where the warps holding those queries put them
                const uint32_t p_col = h * 64 + (k4 >> 1) * 32 + (k4 & 1) * 8;
                const uint32_t ko = ((kk >> 2) * (kT * 128) + (kk & 3) * 32) >> 4;
                const uint32_t mo = (kk * 16 * 128) >> 4;
                if (k4 == 0 && first) {
                    mma_ts_w<0>(tmem + C::COL_DV, tmem + C::COL_ST + p_col, do_mn + mo,
                                C::IDESC_KV);
                    mma_ss_w<0>(tmem + C::COL_DK, ds_d + ko, q_mn + mo, C::IDESC_KV);
                } else {
                    mma_ts_w<1>(tmem + C::COL_DV, tmem + C::COL_ST + p_col, do_mn + mo,
                                C::IDESC_KV);
                    mma_ss_w<1>(tmem + C::COL_DK, ds_d + ko, q_mn + mo, C::IDESC_KV);
                }
            }
        };
        // a wait the whole warp agrees on (the elected issue needs all lanes)
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
        };
        bool ok = wait_all(bar_kv, 0);
        for (int s = 0; s < n_steps && ok; ++s) {
            const uint32_t x = static_cast<uint32_t>(s) & 1u;
            const uint32_t ph = x;
            if (!wait_all(bar_q(x), static_cast<uint32_t>(s >> 1) & 1u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t q_buf = sQ + x * C::TILE_BYTES, o_buf = sDO + x * C::TILE_BYTES;
            // S^T_0 needs no wait: it overwrites only P^T of the previous step,
            // which that step's dV product (issued earlier) has read
            issue_t(C::COL_ST, k_d, q_buf, 0);
            if (s > 0) {
                // dP^T goes over the previous step's dQ: wait until it is read;
                // that step's products are then done, so its buffer takes the
                // next step's Q and dO
                if (!wait_all(bar_dq, ph ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (s + 1 < n_steps) {
                    load_q(s + 1);
                    ++q_loads;
                }
            }
            issue_t(C::COL_DPT, v_d, o_buf, 0);
            mma_commit_w(bar_s0);
            issue_t(C::COL_ST, k_d, q_buf, 1);
            issue_t(C::COL_DPT, v_d, o_buf, 1);
            mma_commit_w(bar_s1);
            if (!wait_all(bar_p0, ph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            issue_kv(0, x, s == 0);
            if (!wait_all(bar_p1, ph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            issue_kv(1, x, false);
            // dQ = dS K over all 128 keys
            mma_ss_w<0>(tmem + C::COL_DQ, ds_mn, k_mn, C::IDESC_Q);
#pragma unroll
            for (int kk = 1; kk < kT / 16; ++kk) {
                const uint32_t mo = (kk * 16 * 128) >> 4;
                mma_ss_w<1>(tmem + C::COL_DQ, ds_mn + mo, k_mn + mo, C::IDESC_Q);
            }
            mma_commit_w(bar_m2);
        }
        if (!ok || *abort) {
            mma_commit_w(bar_drain);
            mbar_wait_drain(bar_drain, 0);
            mbar_wait_drain(bar_kv, 0);
            for (int xb = 0; xb < 2; ++xb) {
                const int n = q_loads / 2 + (xb < q_loads % 2 ? 1 : 0);   // copies into buffer xb
                if (n > 0)
                    mbar_wait_drain(bar_q(xb), static_cast<uint32_t>(n - 1) & 1u);
            }
        }
    } else {
        // ------------------------------------------------------------ compute
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float scale_log2 = a.scale_log2;
        float4 acc[DH / 4];                       // dQ row segment of the previous step
        float4 *acc_dst = nullptr;                // where it goes (null: nothing pending)
        bool ok = true;
        for (int s = 0; s < n_steps && ok; ++s) {
            const uint32_t ph = static_cast<uint32_t>(s) & 1u;
            const int hq = step_hq(s), it = step_it(s);
            {
                // -lse (log2 units) and Delta of the tile's query rows; the
                // previous step's readers are past bar_m2, which needed them all
                const int c = tid & (kT - 1);
                const int i = it * kT + c;
                const size_t row = static_cast<size_t>(q0 + i) * H + hq;
                if (tid < kT)
                    nl_s[c] = i < lq ? -a.lse[row] * kLog2e : 0.f;
                else
                    delta_s[c] = i < lq ? a.delta[row] : 0.f;
            }
            mbar_arrive(bar_ld);
            ok = __all_sync(0xffffffffu, mbar_wait(bar_ld, ph, abort));
            if (!ok)
                break;
            // a tile every (key, query) pair of which is visible needs no mask
            BwdMask m;
            m.j = j;
            m.lk = lk;
            m.lq = lq;
            m.causal = a.causal;
            m.wl = wl;
            m.i_lo = static_cast<long long>(it) * kT;
            m.off = off;
            const bool full = j_lo + kT <= lk && m.i_lo + kT <= lq &&
                              (!a.causal || j_lo + kT - 1 <= m.i_lo + off) &&
                              (wl < 0 || j_lo >= m.i_lo + kT - 1 + off - wl);
            // the query halves in turn, all eight warps on each: this warp takes
            // queries 64 h + 32 g .. +31 of its 32 rows, so the tensor core runs
            // half 1's S^T / dP^T and half 0's dV / dK while it works
#pragma unroll 1
            for (int h = 0; h < 2 && ok; ++h) {
                ok = __all_sync(0xffffffffu, mbar_wait(h ? bar_s1 : bar_s0, ph, abort));
                if (!ok)
                    break;
                tc_fence_after();
                uint32_t pk[16];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int cb = h * 64 + sub * 32 + c2 * 16;   // first query column of the chunk
                    uint32_t sr[16], dr[16];
                    tmem_ld16(tmem + lane_addr + C::COL_ST + cb, sr);
                    tmem_ld16(tmem + lane_addr + C::COL_DPT + cb, dr);
                    tmem_wait_ld();
                    uint32_t dk2[8];
                    if (full)
                        bwd_chunk<true>(sr, dr, scale_log2, sLse, sDelta, cb, m, pk + c2 * 8, dk2);
                    else
                        bwd_chunk<false>(sr, dr, scale_log2, sLse, sDelta, cb, m, pk + c2 * 8, dk2);
#pragma unroll
                    for (int q8 = 0; q8 < 2; ++q8)
                        st_shared_v4(sDS + sw_chunk(r, (cb >> 3) + q8), dk2[4 * q8],
                                     dk2[4 * q8 + 1], dk2[4 * q8 + 2], dk2[4 * q8 + 3]);
                }
                // P^T (bf16 pairs) of these 32 queries over their own S^T columns,
                // which only this warp reads
                tmem_st16(tmem + lane_addr + C::COL_ST + h * 64 + sub * 32, pk);
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(h ? bar_p1 : bar_p0);
            }
            if (!ok)
                break;
            if (acc_dst != nullptr)
                flush_dq<DH>(acc_dst, acc);
            ok = __all_sync(0xffffffffu, mbar_wait(bar_m2, ph, abort));
            if (!ok)
                break;
            tc_fence_after();
            // this half of the q tile's dQ rows (TMEM lane = query row)
#pragma unroll
            for (int cb = 0; cb < DH; cb += 32) {
                uint32_t qr[32];
                tmem_ld32(tmem + lane_addr + C::COL_DQ + half * DH + cb, qr);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    acc[(cb + e) >> 2] =
                        make_float4(__uint_as_float(qr[e]), __uint_as_float(qr[e + 1]),
                                    __uint_as_float(qr[e + 2]), __uint_as_float(qr[e + 3]));
            }
            tc_fence_before();
            mbar_arrive(bar_dq);
            const int i = it * kT + r;
            acc_dst = i < lq ? reinterpret_cast<float4 *>(
                                   a.dq_acc + (static_cast<size_t>(q0 + i) * H + hq) * D +
                                   half * DH)
                             : nullptr;
        }
        if (ok && acc_dst != nullptr)
            flush_dq<DH>(acc_dst, acc);
    }

    tc_fence_before();
    __syncthreads();
    if (*abort == 0 && warp < kComputeWarps) {
        // dK (scaled) and dV rows of this key tile, this thread's column half
        tc_fence_after();
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float sc = a.scale;
        const size_t row = (static_cast<size_t>(k0 + j) * Hkv + kh) * D + half * DH;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            const uint32_t col = (which == 0 ? C::COL_DV : C::COL_DK) + half * DH;
            const float f = which == 0 ? 1.f : sc;
            __nv_bfloat16 *dst = which == 0 ? dv : dk;
#pragma unroll
            for (int cb = 0; cb < DH; cb += 32) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_addr + col + cb, rr);
                tmem_wait_ld();
                if (j < lk) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(rr[e]) * f, __uint_as_float(rr[e + 1]) * f);
                        v.y = pack_bf16x2(__uint_as_float(rr[e + 2]) * f,
                                          __uint_as_float(rr[e + 3]) * f);
                        v.z = pack_bf16x2(__uint_as_float(rr[e + 4]) * f,
                                          __uint_as_float(rr[e + 5]) * f);
                        v.w = pack_bf16x2(__uint_as_float(rr[e + 6]) * f,
                                          __uint_as_float(rr[e + 7]) * f);
                        *reinterpret_cast<uint4 *>(dst + row + cb + e) = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort && tid == 0)
        atomicCAS(a.status, VFA_OK, VFA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------ dQ

template <int D>
__global__ void bwd_dq_kernel(const BwdArgs a)
{
    if (*a.status != VFA_OK)
        return;
    const long long n4 = static_cast<long long>(a.total_q) * a.num_heads * D / 4;
    const float sc = a.scale;
    const float4 *src = reinterpret_cast<const float4 *>(a.dq_acc);
    uint2 *dst = reinterpret_cast<uint2 *>(a.dq);
    for (long long x = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; x < n4;
         x += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 v = src[x];
        dst[x] = make_uint2(pack_bf16x2(v.x * sc, v.y * sc), pack_bf16x2(v.z * sc, v.w * sc));
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs &a, int key_tile_bound, int sm_count, cudaStream_t s)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(BwdCfg<D>::SMEM));
        if (e != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    bwd_prep_kernel<<<1, kPrepThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    const int grid_rows = sm_count * 8;
    bwd_delta_kernel<D><<<grid_rows, 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    if (key_tile_bound > 0) {
        bwd_kernel<D><<<dim3(key_tile_bound, a.num_kv_heads), kThreads, BwdCfg<D>::SMEM, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    bwd_dq_kernel<D><<<grid_rows, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(int batch, int total_q, int num_heads, int head_dim)
{
    size_t n = 256;                                                   // status word
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);          // key tile starts
    n = (n + 255) & ~static_cast<size_t>(255);
    n += static_cast<size_t>(total_q) * num_heads * sizeof(float);    // Delta
    n = (n + 255) & ~static_cast<size_t>(255);
    n += static_cast<size_t>(total_q) * num_heads * head_dim * sizeof(float);   // dQ sum
    return (n + 255) & ~static_cast<size_t>(255);
}

void bwd_workspace_split(void *ws, int batch, int total_q, int num_heads, BwdArgs *a)
{
    uint8_t *p = static_cast<uint8_t *>(ws);
    a->status = reinterpret_cast<int32_t *>(p);
    size_t n = 256;
    a->ktile_start = reinterpret_cast<int32_t *>(p + n);
    n += (static_cast<size_t>(batch) + 1) * sizeof(int32_t);
    n = (n + 255) & ~static_cast<size_t>(255);
    a->delta = reinterpret_cast<float *>(p + n);
    n += static_cast<size_t>(total_q) * num_heads * sizeof(float);
    n = (n + 255) & ~static_cast<size_t>(255);
    a->dq_acc = reinterpret_cast<float *>(p + n);
}

cudaError_t launch_bwd(int head_dim, const BwdArgs &a, int key_tile_bound, int sm_count,
                       cudaStream_t stream)
{
    switch (head_dim) {
    case 64: return launch_bwd_d<64>(a, key_tile_bound, sm_count, stream);
    case 128: return launch_bwd_d<128>(a, key_tile_bound, sm_count, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vfa
