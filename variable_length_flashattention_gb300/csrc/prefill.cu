// prefill.cu -- variable-length attention forward on sm_103a, one q tile per
// CTA work item (used for head_dim 256, whose O accumulator alone fills half
// of TMEM; head_dim 64 and 128 use prefill_pair.cu).  An FP8 instantiation
// takes Q and K as E4M3 codes: their tiles are half the bytes and S = Q K^T
// runs as kind::f8f6f4 in 32-byte k-steps (the per-tensor descales are
// folded into the score scale); P, V and O are the bf16 kernel's.
//
// Computes, per packed query row, softmax(scale * q K^T, masks) V and the
// natural-log log-sum-exp, by the tiled online-softmax recurrence of
// "Varlen Flash Attention Implementation Plan", Task 1 Step 1 (running row
// max m, running denominator l, accumulator rescaled when m grows, final
// out = acc / l, lse = m + log l; causal and sequence-boundary masks on local
// positions).  The plan's tile sizes, thread layout and sequence lookup are
// not kept; this kernel is built for Blackwell:
//
//   * persistent CTAs take (sequence, 128-row q tile, head) items from the
//     device-built work list (sched.cu) through an atomic counter; the
//     producer warp fetches and hands each item to the other warps through a
//     two-slot shared-memory ring;
//   * warp 0 moves Q, K and V tiles with TMA (128-byte swizzle) into a
//     shared-memory ring guarded by mbarriers;
//   * warp 1 issues tcgen05.mma: S = Q K^T into one of three TMEM buffers, and
//     O += P V with P read straight from TMEM (P overwrites its S buffer as
//     bf16) and V as an MN-major shared-memory operand;
//   * warps 2-5 own one query row per thread: they read S rows from TMEM,
//     take the row max on the raw scores (the scale is positive), fold scale
//     and max into one FMA before exp2, keep m and l, write P back to TMEM,
//     rescale O in TMEM only when the row max has grown by more than 2^8
//     (exact after the final division because l and O always share one
//     reference max), and run the epilogue (O / l -> bf16, lse).
// Every wait is bounded: on expiry the kernel records VFA_ERR_TIMEOUT,
// drains its own in-flight copies and MMAs, frees TMEM and returns.
#include <cfloat>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

// F8: Q and K are FP8 E4M3 codes (1 byte each) and S = Q K^T runs as
// kind::f8f6f4 in 32-byte k-steps; V, P and O stay as in the bf16 kernel.
template <int D, bool F8 = false>
struct Cfg {
    static constexpr int BQ = kBlockQ;
    static constexpr int BK = block_k_for(D);
    static constexpr int NS = 2;                          // K/V ring stages
    static constexpr int NQ = D == 256 ? 1 : 2;           // Q buffers
    static constexpr int DB = D / 64;                     // 128-byte column blocks per V / O row
    static constexpr int QK_ELEM = F8 ? 1 : 2;            // bytes per Q / K element
    static constexpr int QK_DB = D * QK_ELEM / 128;       // 128-byte column blocks per Q / K row
    static constexpr int QK_BLOCK = 128 / QK_ELEM;        // elements per such block
    static constexpr int KSTEPS = D * QK_ELEM / 32;       // 32-byte MMA k-steps of S = Q K^T
    static constexpr uint32_t Q_BYTES = BQ * D * QK_ELEM;
    static constexpr uint32_t K_BYTES = BK * D * QK_ELEM;
    static constexpr uint32_t KV_BYTES = BK * D * 2;      // one V stage
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSB = 3;                         // S/P buffers in TMEM
    static constexpr uint32_t O_COL = 0;                  // O: columns [0, D)
    static constexpr uint32_t S_COL = D;                  // S buffer x: [D + x*BK, D + (x+1)*BK)
    static constexpr int NUM_BARS = 2 * NQ + 4 * NS + 3 * NSB + 1 + 4;
    static constexpr size_t SMEM = 1024 /*alignment slack*/ + NQ * Q_BYTES +
                                   NS * (K_BYTES + KV_BYTES) + NUM_BARS * 8 + 64;
    static constexpr uint32_t IDESC_QK =
        F8 ? idesc_e4m3_f32(BQ, BK) : idesc_bf16_f32(BQ, BK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BQ, D, false, true);
    static_assert(S_COL + NSB * BK <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

constexpr int kThreads = 192;      // 6 warps: TMA, MMA, 4 x softmax/epilogue
constexpr int kItemConsumers = 5;  // MMA lane + one arrival per softmax warp

__device__ __forceinline__ void record_error(int32_t *status, int code)
{
    atomicCAS(status, 0, code);
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs p)
{
    using C = Cfg<D, F8>;
    constexpr int BQ = C::BQ, BK = C::BK, NS = C::NS, NQ = C::NQ, DB = C::DB;

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    // (b, i, h, end key tile), (q row 0 of b, Lq, Lk, k row 0 of b), (first key tile, -, -, -)
    __shared__ int4 s_item[2][3];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // 1024-byte aligned carve-up (128-byte swizzle atoms need it).
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sQ = base;
    const uint32_t sK = sQ + NQ * C::Q_BYTES;
    const uint32_t sV = sK + NS * C::K_BYTES;
    const uint32_t bars = sV + NS * C::KV_BYTES;
    auto q_full = [&](int i) { return bars + 8u * i; };
    auto q_empty = [&](int i) { return bars + 8u * (NQ + i); };
    auto k_full = [&](int i) { return bars + 8u * (2 * NQ + i); };
    auto k_empty = [&](int i) { return bars + 8u * (2 * NQ + NS + i); };
    auto v_full = [&](int i) { return bars + 8u * (2 * NQ + 2 * NS + i); };
    auto v_empty = [&](int i) { return bars + 8u * (2 * NQ + 3 * NS + i); };
    constexpr int NSB = C::NSB;
    auto s_full = [&](int x) { return bars + 8u * (2 * NQ + 4 * NS + x); };
    auto s_free = [&](int x) { return bars + 8u * (2 * NQ + 4 * NS + NSB + x); };
    auto p_full = [&](int x) { return bars + 8u * (2 * NQ + 4 * NS + 2 * NSB + x); };
    const uint32_t drain_bar = bars + 8u * (2 * NQ + 4 * NS + 3 * NSB);
    auto item_full = [&](int x) { return bars + 8u * (2 * NQ + 4 * NS + 3 * NSB + 1 + x); };
    auto item_empty = [&](int x) { return bars + 8u * (2 * NQ + 4 * NS + 3 * NSB + 3 + x); };
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NQ; ++i) {
            mbar_init(q_full(i), 1);
            mbar_init(q_empty(i), 1);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
        }
        for (int x = 0; x < NSB; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(s_free(x), 1);
            mbar_init(p_full(x), 128);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(item_full(x), 1);
            mbar_init(item_empty(x), kItemConsumers);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    // The work list is written by the scheduler grid launched just before.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Take the next item from the ring (consumer side); false at the end.
    // The item visits key tiles [first, it.w).
    auto next_item = [&](uint32_t n, int4 &it, int4 &seq, int &first) -> bool {
        const int slot = n & 1;
        if (!mbar_wait(item_full(slot), (n >> 1) & 1u, abort))
            return false;
        it = s_item[slot][0];
        seq = s_item[slot][1];
        first = s_item[slot][2].x;
        return it.x >= 0;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int n_items = (*p.status == 0) ? *p.n_items : 0;
            uint32_t n = 0, qit = 0, kfills = 0, vfills = 0;
            bool ok = true;
            for (;; ++n) {
                const int slot = n & 1;
                if (!mbar_wait(item_empty(slot), ((n >> 1) & 1u) ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                const int idx = atomicAdd(p.next_item, 1);
                const int4 it = idx < n_items ? p.items[2 * idx] : make_int4(-1, 0, 0, 0);
                int4 seq = make_int4(0, 0, 0, 0);
                int first = 0;
                if (it.x >= 0) {
                    const int q0 = p.cu_q[it.x], k0 = p.cu_k[it.x];
                    seq = make_int4(q0, p.cu_q[it.x + 1] - q0, p.cu_k[it.x + 1] - k0, k0);
                    first = p.items[2 * idx + 1].z;
                }
                s_item[slot][0] = it;
                s_item[slot][1] = seq;
                s_item[slot][2] = make_int4(first, 0, 0, 0);
                mbar_arrive(item_full(slot));
                if (it.x < 0)
                    break;
                const int i = it.y, h = it.z, j_end = it.w;
                if (j_end <= first)
                    continue;
                const int q_row0 = seq.x + i * BQ;
                const int k_row0 = seq.w;
                const int qb = qit % NQ;
                if (!mbar_wait(q_empty(qb), ((qit / NQ) & 1u) ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(q_full(qb), C::Q_BYTES);
                for (int db = 0; db < C::QK_DB; ++db)
                    tma_load_3d(sQ + qb * C::Q_BYTES + db * (BQ * 128), &p.tm_q, q_full(qb),
                                db * C::QK_BLOCK, h, q_row0);
                ++qit;
                for (int j = first; j < j_end; ++j) {
                    const int st = kfills % NS;
                    if (!mbar_wait(k_empty(st), ((kfills / NS) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full(st), C::K_BYTES);
                    for (int db = 0; db < C::QK_DB; ++db)
                        tma_load_3d(sK + st * C::K_BYTES + db * (BK * 128), &p.tm_k, k_full(st),
                                    db * C::QK_BLOCK, h / p.kv_group, k_row0 + j * BK);
                    ++kfills;
                    if (!mbar_wait(v_empty(st), ((vfills / NS) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full(st), C::KV_BYTES);
                    for (int db = 0; db < DB; ++db)
                        tma_load_3d(sV + st * C::KV_BYTES + db * (BK * 128), &p.tm_v, v_full(st),
                                    db * 64, h / p.kv_group, k_row0 + j * BK);
                    ++vfills;
                }
                if (!ok)
                    break;
            }
            if (!ok || *abort) {
                // Drain: the last fill of each stage / Q buffer may still be in flight.
                auto last_fill_wait = [&](uint32_t fills, int nslots, int slot, uint32_t bar) {
                    const uint32_t k = fills / nslots + (static_cast<uint32_t>(slot) < fills % nslots ? 1u : 0u);
                    if (k > 0)
                        mbar_wait_drain(bar, (k - 1) & 1u);
                };
                for (int st = 0; st < NS; ++st) {
                    last_fill_wait(kfills, NS, st, k_full(st));
                    last_fill_wait(vfills, NS, st, v_full(st));
                }
                for (int qb = 0; qb < NQ; ++qb)
                    last_fill_wait(qit, NQ, qb, q_full(qb));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // All 32 lanes run this loop on warp-uniform values (operands in
        // uniform registers); one elected lane issues each MMA and commit.
        {
            // Descriptors of every buffer, built once; a k-step only adds a
            // compile-time offset (in 16-byte units) to the start-address field.
            // (The start-address field is the low 14 bits, address / 16; shared
            // addresses stay below 256 KiB, so descriptors are linear in it.)
            const uint64_t q_desc0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t k_desc0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t v_desc0 = sdesc_sw128(sV, BK * 128, 1024);
            uint32_t n = 0, qit = 0, kv = 0, g = 0;
            bool ok = true;
            // O += P V for the key tile with global index gp held in ring slot kvp.
            auto issue_pv = [&](uint32_t gp, uint32_t kvp, bool acc) -> bool {
                const int xp = gp % NSB;
                const int stp = kvp % NS;
                if (!mbar_wait(p_full(xp), (gp / NSB) & 1u, abort))
                    return false;
                if (!mbar_wait(v_full(stp), (kvp / NS) & 1u, abort))
                    return false;
                tc_fence_after();
                const uint64_t vd = v_desc0 + stp * (C::KV_BYTES >> 4);
                const uint32_t a_tm = tmem + C::S_COL + xp * BK;
                if (acc)
                    mma_ts_w<1>(tmem + C::O_COL, a_tm, vd, C::IDESC_PV);
                else
                    mma_ts_w<0>(tmem + C::O_COL, a_tm, vd, C::IDESC_PV);
#pragma unroll
                for (int kk = 1; kk < BK / 16; ++kk)
                    mma_ts_w<1>(tmem + C::O_COL, a_tm + kk * 8, vd + kk * (16 * 128 / 16),
                                C::IDESC_PV);
                mma_commit_w(s_free(xp));
                mma_commit_w(v_empty(stp));
                return true;
            };
            for (;; ++n) {
                int4 it, seq;
                int first;
                const bool more = next_item(n, it, seq, first);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(item_empty(n & 1));
                if (!more)
                    break;
                const int j_end = it.w;
                if (j_end <= first)
                    continue;
                const int qb = qit % NQ;
                if (!mbar_wait(q_full(qb), (qit / NQ) & 1u, abort)) {
                    ok = false;
                    break;
                }
                const uint64_t qd = q_desc0 + qb * (C::Q_BYTES >> 4);
                for (int j = first; j < j_end; ++j) {
                    const int st = kv % NS;
                    const int x = g % NSB;
                    if (!mbar_wait(k_full(st), (kv / NS) & 1u, abort) ||
                        !mbar_wait(s_free(x), ((g / NSB) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kd = k_desc0 + st * (C::K_BYTES >> 4);
                    const uint32_t s_tm = tmem + C::S_COL + x * BK;
                    // k-steps of 32 bytes: 16 bf16 or 32 FP8 elements
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS; ++kk) {
                        const uint64_t qo = qd + (((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4);
                        const uint64_t ko = kd + (((kk >> 2) * (BK * 128) + (kk & 3) * 32) >> 4);
                        if constexpr (F8) {
                            if (kk == 0)
                                mma_ss_w8<0>(s_tm, qo, ko, C::IDESC_QK);
                            else
                                mma_ss_w8<1>(s_tm, qo, ko, C::IDESC_QK);
                        } else {
                            if (kk == 0)
                                mma_ss_w<0>(s_tm, qo, ko, C::IDESC_QK);
                            else
                                mma_ss_w<1>(s_tm, qo, ko, C::IDESC_QK);
                        }
                    }
                    mma_commit_w(s_full(x));
                    mma_commit_w(k_empty(st));
                    if (j == j_end - 1)
                        mma_commit_w(q_empty(qb));
                    if (j > first && !issue_pv(g - 1, kv - 1, j - 1 > first)) {
                        ok = false;
                        break;
                    }
                    ++g;
                    ++kv;
                }
                if (!ok)
                    break;
                if (!issue_pv(g - 1, kv - 1, j_end - 1 > first)) {
                    ok = false;
                    break;
                }
                ++qit;
            }
            if (!ok || *abort) {
                // Every MMA this warp issued must finish before TMEM is freed.
                mma_commit_w(drain_bar);
                mbar_wait_drain(drain_bar, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int quarter = warp & 3;                 // TMEM lanes [32*quarter, 32*quarter+32)
        const int r = quarter * 32 + lane;            // this thread's row in the q tile
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const float scale_log2 = p.scale_log2;
        const int H = p.num_heads;
        uint32_t g = 0;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

        const float2 scale2 = make_float2(scale_log2, scale_log2);
        for (uint32_t n = 0;; ++n) {
            int4 it, seq;
            int first;
            const bool more = next_item(n, it, seq, first);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(item_empty(n & 1));
            if (!more)
                break;
            const int i = it.y, h = it.z, j_end = it.w;
            const int q0 = seq.x, lq = seq.y, lk = seq.z;
            const int q_local = i * BQ + r;
            const bool row_valid = q_local < lq;
            const long long tok = static_cast<long long>(q0) + q_local;

            if (j_end <= first) {
                if (row_valid) {
                    uint4 z = make_uint4(0, 0, 0, 0);
                    uint4 *dst = reinterpret_cast<uint4 *>(out + (tok * H + h) * D);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c)
                        dst[c] = z;
                    p.lse[tok * H + h] = -FLT_MAX;
                }
                continue;
            }

            float m_used = -INFINITY;     // reference max, log2 units of the scaled score
            float l = 0.f;
            bool ok = true;
            for (int j = first; j < j_end; ++j) {
                const int x = g % NSB;
                if (!mbar_wait(s_full(x), (g / NSB) & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_addr + C::S_COL + x * BK;
                float s[BK];
                {
                    uint32_t sr[BK];
#pragma unroll
                    for (int c = 0; c < BK / 32; ++c)
                        tmem_ld32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < BK; ++c)
                        s[c] = __uint_as_float(sr[c]);
                }
                // Row max of the raw scores (the scale is positive): eight
                // independent three-input max chains.
                const int k_base = j * BK;
                // causal: row q sees keys <= q + off (off = 0 top-left, Lk - Lq
                // bottom-right); a window also hides keys < q + off - window_left
                const int off = p.causal == 2 ? lk - lq : 0;
                const int wl = p.window_left;
                const bool need_lo =
                    wl >= 0 && k_base < static_cast<long long>(i) * BQ + BQ - 1 + off - wl;
                const bool need_mask = need_lo || (k_base + BK > lk) ||
                                       (p.causal && k_base + BK - 1 > i * BQ + off);
                if (need_mask) {
                    // keys in [lo, lim) visible
                    const int lim = (p.causal ? min(lk, max(0, q_local + off + 1)) : lk) - k_base;
                    const int lo = need_lo ? static_cast<int>(min(
                                                 static_cast<long long>(BK),
                                                 max(0ll, static_cast<long long>(q_local) + off -
                                                              wl - k_base)))
                                           : 0;
#pragma unroll
                    for (int c = 0; c < BK; ++c)
                        s[c] = (c < lim && c >= lo) ? s[c] : -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    mx[e] = fmaxf(s[e], s[e + 8]);
#pragma unroll
                for (int c = 16; c < BK; c += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        mx[e] = fmax3(mx[e], s[c + e], s[c + 8 + e]);
                const float mt_raw = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                           fmaxf(mx[6], mx[7]));
                const float m_tile = mt_raw == -INFINITY ? -INFINITY : mt_raw * scale_log2;
                const float m_new = fmaxf(m_used, m_tile);
                const bool grow = m_new > m_used + 8.0f;    // also true for m_used = -inf
                if (j == first) {
                    m_used = m_new;
                } else if (__any_sync(0xffffffffu, grow)) {
                    // O must hold the previous tile's product before it is rescaled.
                    const uint32_t gp = g - 1;
                    if (!mbar_wait(s_free(gp % NSB), (gp / NSB) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float f = (m_new == -INFINITY) ? 1.f : ex2_approx(m_used - m_new);
                    const uint32_t o_addr = tmem + lane_addr + C::O_COL;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t rr[32];
                        tmem_ld32(o_addr + c * 32, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            rr[e] = __float_as_uint(__uint_as_float(rr[e]) * f);
                        tmem_st32(o_addr + c * 32, rr);
                    }
                    tmem_wait_st();
                    l *= f;
                    m_used = m_new;
                }
                // p = 2^(s * scale_log2 - m): packed FMA pairs, one exp2 per score,
                // packed sums into four pair accumulators.
                const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
                const float2 negm2 = make_float2(neg_m, neg_m);
                float2 ls[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    ls[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < BK / 64; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float2 t = __ffma2_rn(make_float2(s[c * 64 + 2 * e], s[c * 64 + 2 * e + 1]),
                                                    scale2, negm2);
                        const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                        ls[e & 3] = __fadd2_rn(ls[e & 3], pp);
                        pk[e] = pack_bf16x2(pp.x, pp.y);
                    }
                    tmem_st32(s_addr + c * 32, pk);
                }
                const float2 l2 = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
                l += l2.x + l2.y;
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full(x));
                ++g;
            }
            if (!ok)
                break;

            // Epilogue: wait for the item's last O += P V, then O / l -> bf16 and lse.
            const uint32_t gl = g - 1;
            if (!mbar_wait(s_free(gl % NSB), (gl / NSB) & 1u, abort))
                break;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const uint32_t o_addr = tmem + lane_addr + C::O_COL;
            uint4 *dst = reinterpret_cast<uint4 *>(out + (tok * H + h) * D);
            // 128 columns of O per TMEM wait (the wait covers all of a thread's
            // loads in flight, so smaller pieces would each expose its latency)
#pragma unroll
            for (int c0 = 0; c0 < D / 32; c0 += 4) {
                uint32_t rr[4][32];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld32(o_addr + (c0 + q) * 32, rr[q]);
                tmem_wait_ld_r(rr[0]);
                tmem_bind_r(rr[1]);
                tmem_bind_r(rr[2]);
                tmem_bind_r(rr[3]);
                if (row_valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(rr[q][8 * e + 0]) * inv_l,
                                              __uint_as_float(rr[q][8 * e + 1]) * inv_l);
                            v.y = pack_bf16x2(__uint_as_float(rr[q][8 * e + 2]) * inv_l,
                                              __uint_as_float(rr[q][8 * e + 3]) * inv_l);
                            v.z = pack_bf16x2(__uint_as_float(rr[q][8 * e + 4]) * inv_l,
                                              __uint_as_float(rr[q][8 * e + 5]) * inv_l);
                            v.w = pack_bf16x2(__uint_as_float(rr[q][8 * e + 6]) * inv_l,
                                              __uint_as_float(rr[q][8 * e + 7]) * inv_l);
                            dst[(c0 + q) * 4 + e] = v;
                        }
                    }
                }
            }
            if (row_valid)
                p.lse[tok * H + h] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -FLT_MAX;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 0)
        record_error(p.status, VFA_ERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool F8>
cudaError_t launch_d(const PrefillArgs &a, int grid, cudaStream_t stream)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(prefill_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Cfg<D, F8>::SMEM));
        if (e != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    // Programmatic dependent launch: the prologue overlaps the scheduler grid.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<D, F8>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_kernel<D, F8>, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(int head_dim, const PrefillArgs &a, int grid, cudaStream_t stream)
{
    if (pairs_for(head_dim))
        return launch_prefill_pair(head_dim, a, grid, stream);
    if (head_dim == 256)
        return a.qk_fp8 ? launch_d<256, true>(a, grid, stream)
                        : launch_d<256, false>(a, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace vfa
