// prefill_pair.cu -- variable-length attention forward on sm_103a, two q
// tiles per CTA work item (head_dim 64 and 128).
//
// Same definition as prefill.cu ("Varlen Flash Attention Implementation
// Plan", Task 1 Step 1: scaled scores, causal and key-boundary masks on local
// positions, online softmax with running max m and denominator l, out =
// acc / l, lse = m + log l).  What changes is how the work is laid out on
// the SM:
//
//   * a work item holds two q tiles (a, b) of the same (sequence, head); each
//     K/V tile is loaded once by TMA and used by both;
//   * warp 0 loads Q and K, warp 2 loads V, each with its own ring; that
//     warpgroup hands registers to the softmax warpgroups (setmaxnreg);
//   * warp 1 issues, per key tile j:  S_a = Q_a K_j^T,  O_b += P_b V_{j-1},
//     S_b = Q_b K_j^T,  O_a += P_a V_j  -- while one softmax warpgroup works
//     on its scores the tensor core runs the other tile's products.  P_x
//     lives in S_x's TMEM columns; the next S_x is issued right after the
//     O_x += P_x V that reads it: tcgen05.mma instructions of one thread run
//     in issue order, so the product has read P_x before S_x is rewritten
//     (and waiting for its completion instead would idle the tensor core);
//   * warps 4-7 own tile a's 128 rows, warps 8-11 tile b's, one row per
//     thread (TMEM lane = row).  A key tile's 128 scores of a row come into
//     registers with one TMEM wait (tcgen05.wait::ld waits for all of a
//     thread's loads, so loading in pieces would expose the load latency once
//     per piece); the row max is taken from the registers, the reference max
//     moves (O, l rescaled) only if the tile's max exceeds it by more than
//     2^8, and p is then computed once per score.  Each half of P (64 keys)
//     is published on its own and O_x += P_x V runs per half, so the tensor
//     core starts on the first 64 keys while the second half is still being
//     exponentiated;
//   * in a masked tile (causal diagonal, ragged key tail) a 32-column chunk
//     that is valid for all 32 rows of a warp skips the mask, and one that
//     is masked for all of them skips its exponentials;
//   * O / l leaves through a 2 KB shared-memory stage per warp (no cross-warp
//     handshake): a warp whose 32 rows all lie in the sequence hands each
//     32-column chunk to a TMA tile store; in a sequence's last tile, plain
//     stores write eight whole 64-byte row segments per instruction;
//   * TMEM: O_a, O_b (D columns each), S/P_a, S/P_b (128 columns each);
//   * an FP8 instantiation takes Q and K as E4M3 codes: their tiles are half
//     the bytes (at head_dim 64 rows of 64 bytes, stored with the 64-byte
//     swizzle) and S = Q K^T runs as kind::f8f6f4 in 32-byte k-steps; the
//     per-tensor descales are folded into the score scale.
// Everything else (item ring fed by an atomic counter, bounded waits with
// drain-and-report on expiry) is as in prefill.cu.
#include <cfloat>
#include <type_traits>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

// F8: Q and K are FP8 E4M3 codes (1 byte each) and S = Q K^T runs as
// kind::f8f6f4; V, P and O stay as in the bf16 kernel.
template <int D, bool F8 = false>
struct PairCfg {
    static constexpr int BQ = kBlockQ;
    static constexpr int BK = 128;
    static constexpr int NS = D == 64 ? 4 : 2;            // K and V ring stages
    static constexpr int DB = D / 64;                     // 128-byte column blocks per V / O row
    static constexpr int QK_ELEM = F8 ? 1 : 2;            // bytes per Q / K element
    // Q / K rows are stored in swizzled column blocks of QK_ROW bytes: 128
    // (128-byte swizzle), or 64 for FP8 at head_dim 64, whose rows are only 64
    // bytes (64-byte swizzle)
    static constexpr int QK_ROW = D * QK_ELEM >= 128 ? 128 : 64;
    static constexpr int QK_DB = D * QK_ELEM / QK_ROW;    // column blocks per Q / K row
    static constexpr int QK_BLOCK = QK_ROW / QK_ELEM;     // elements per such block
    static constexpr int QK_KSTEP = 32 / QK_ELEM;         // elements per MMA k-step (32 bytes)
    static constexpr uint32_t Q_BYTES = BQ * D * QK_ELEM;
    static constexpr uint32_t K_BYTES = BK * D * QK_ELEM;
    static constexpr uint32_t KV_BYTES = BK * D * 2;      // one V stage
    static constexpr uint32_t WARP_STAGE = 32 * 64;       // one warp's 32 rows x 32 output columns
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 2 * D;              // S_x at S_COL + x * BK; O_x at x * D
    static constexpr int NUM_BARS = 4 + 4 * NS + 15;
    static constexpr size_t SMEM = 1024 + 2 * Q_BYTES + NS * (K_BYTES + KV_BYTES) +
                                   8 * WARP_STAGE + NUM_BARS * 8 + 64;
    static constexpr uint32_t IDESC_QK =
        F8 ? idesc_e4m3_f32(BQ, BK) : idesc_bf16_f32(BQ, BK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BQ, D, false, true);
    static_assert(S_COL + 2 * BK <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// Three warpgroups: warps 0-3 load Q/K (0), issue MMAs (1), load V (2) and
// idle (3); warps 4-7 run tile a's softmax, warps 8-11 tile b's.  The first
// group gives registers up to the two softmax groups (setmaxnreg): 384
// threads launch with 168 registers each, 128 * 120 + 256 * 192 = 384 * 168.
constexpr int kThreads = 384;
constexpr int kVWarp = 2;
constexpr int kFirstMathWarp = 4;
constexpr int kLoadRegs = 120;
constexpr int kMathRegs = 192;
constexpr int kItemConsumers = 10;  // MMA + V loader + one arrival per softmax warp
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale when the max grows by > 2^8

// Masks one 32-column chunk of scores (columns cb..cb+31 of the key tile):
// a row's visible columns are [lo, lim), and scores outside become -inf, so
// they drop out of the max and 2^(-inf) = 0 (the scale is > 0, so no
// -inf * 0).  lim_lo / lo_hi are the warp's smallest lim and largest lo: a
// chunk inside [lo_hi, lim_lo) needs no mask.  LO: a sliding window's edge
// can cut into the tile (otherwise lo = 0).
template <bool LO>
__device__ __forceinline__ void mask_chunk(uint32_t (&sr)[32], int cb, int lim, int lim_lo, int lo,
                                           int lo_hi)
{
    if (cb + 32 <= lim_lo && (!LO || cb >= lo_hi))
        return;
#pragma unroll
    for (int e = 0; e < 32; ++e)
        sr[e] = (cb + e < lim && (!LO || cb + e >= lo)) ? sr[e] : __float_as_uint(-INFINITY);
}

// O rows *= f for this warp's 32 lanes, 16 columns at a time (rare path).
template <int D>
__device__ __forceinline__ void rescale_rows(uint32_t o_addr, float f)
{
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
        uint32_t rr[16];
        tmem_ld16(o_addr + c * 16, rr);
        tmem_wait_ld_r16(rr);
#pragma unroll
        for (int e = 0; e < 16; ++e)
            rr[e] = __float_as_uint(__uint_as_float(rr[e]) * f);
        tmem_st16(o_addr + c * 16, rr);
    }
    tmem_wait_st();
}

// The key tiles of one work item: slot x (0 = tile a, 1 = tile b) visits
// [first[x], end[x]) (empty when end <= first), and the item loads the union
// [j0, j1) of the non-empty ranges, which the scheduler keeps contiguous.
struct ItemSpan {
    int first[2], end[2];
    int j0, j1;
    __device__ __forceinline__ bool live(int x) const { return end[x] > first[x]; }
    __device__ __forceinline__ bool has(int x, int j) const { return j >= first[x] && j < end[x]; }
};

__device__ __forceinline__ ItemSpan item_span(const int4 &it, const int4 &itb)
{
    ItemSpan sp;
    const bool has_b = itb.x >= 0;
    sp.first[0] = itb.z;
    sp.end[0] = it.w;
    sp.first[1] = has_b ? itb.w : 0;
    sp.end[1] = has_b ? itb.y : 0;
    sp.j0 = 0;
    sp.j1 = 0;
    bool any = false;
#pragma unroll
    for (int x = 0; x < 2; ++x)
        if (sp.live(x)) {
            sp.j0 = any ? min(sp.j0, sp.first[x]) : sp.first[x];
            sp.j1 = any ? max(sp.j1, sp.end[x]) : sp.end[x];
            any = true;
        }
    return sp;
}

template <int D, bool WIN, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillArgs p)
{
    using C = PairCfg<D, F8>;
    constexpr int BQ = C::BQ, BK = C::BK, NS = C::NS, DB = C::DB;

    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int4 s_item[2][3];     // (b, i_a, h, cost_a), (i_b, cost_b, -, -), (q0, Lq, Lk, k0)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sQ = base;                           // Q_a, Q_b
    const uint32_t sK = sQ + 2 * C::Q_BYTES;
    const uint32_t sV = sK + NS * C::K_BYTES;
    const uint32_t sO = sV + NS * C::KV_BYTES;          // output staging, 2 KB per softmax warp
    const uint32_t bars = sO + 8 * C::WARP_STAGE;
    auto q_full = [&](int x) { return bars + 8u * x; };
    auto q_empty = [&](int x) { return bars + 8u * (2 + x); };
    auto k_full = [&](int i) { return bars + 8u * (4 + i); };
    auto k_empty = [&](int i) { return bars + 8u * (4 + NS + i); };
    auto v_full = [&](int i) { return bars + 8u * (4 + 2 * NS + i); };
    auto v_empty = [&](int i) { return bars + 8u * (4 + 3 * NS + i); };
    constexpr uint32_t E = 4 + 4 * NS;
    auto s_full = [&](int x) { return bars + 8u * (E + x); };
    // O_x += P_x V runs in two halves of 64 keys; o_h1 / o_h2 complete once
    // per key tile each, when the half's products are in O_x.
    auto o_h1 = [&](int x) { return bars + 8u * (E + 2 + x); };
    auto o_h2 = [&](int x) { return bars + 8u * (E + 4 + x); };
    auto p_half = [&](int x, int hh) { return bars + 8u * (E + 6 + 2 * x + hh); };   // P_x half ready
    auto item_full = [&](int x) { return bars + 8u * (E + 10 + x); };
    auto item_empty = [&](int x) { return bars + 8u * (E + 12 + x); };
    const uint32_t drain_bar = bars + 8u * (E + 14);
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int x = 0; x < 2; ++x) {
            mbar_init(q_full(x), 1);
            mbar_init(q_empty(x), 1);
            mbar_init(s_full(x), 1);
            mbar_init(o_h1(x), 1);
            mbar_init(o_h2(x), 1);
            mbar_init(p_half(x, 0), 128);
            mbar_init(p_half(x, 1), 128);
            mbar_init(item_full(x), 1);
            mbar_init(item_empty(x), kItemConsumers);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
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

    auto next_item = [&](uint32_t n, int4 &it, int4 &itb, int4 &seq) -> bool {
        const int slot = n & 1;
        if (!mbar_wait(item_full(slot), (n >> 1) & 1u, abort))
            return false;
        it = s_item[slot][0];
        itb = s_item[slot][1];
        seq = s_item[slot][2];
        return it.x >= 0;
    };
    // Drain after an abort: the last fill of each ring slot may still be in flight.
    auto last_fill_wait = [&](uint32_t fills, int nslots, int slot, uint32_t bar) {
        const uint32_t k = fills / nslots + (static_cast<uint32_t>(slot) < fills % nslots ? 1u : 0u);
        if (k > 0)
            mbar_wait_drain(bar, (k - 1) & 1u);
    };

    if (warp < kFirstMathWarp) {
    // Each role's code sits inside its setmaxnreg branch, so the register
    // allocator gives it that branch's budget.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLoadRegs));
    if (warp == 0) {
        // ------------------------------------------------------------ items, Q and K
        if (lane == 0) {
            const int n_items = (*p.status == 0) ? *p.n_items : 0;
            uint32_t n = 0, qloads[2] = {0, 0}, kfills = 0;
            bool ok = true;
            for (;; ++n) {
                const int slot = n & 1;
                if (!mbar_wait(item_empty(slot), ((n >> 1) & 1u) ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                const int idx = atomicAdd(p.next_item, 1);
                int4 it = make_int4(-1, 0, 0, 0), itb = make_int4(-1, 0, 0, 0);
                int4 seq = make_int4(0, 0, 0, 0);
                if (idx < n_items) {
                    it = p.items[2 * idx];
                    itb = p.items[2 * idx + 1];
                    const int q0 = p.cu_q[it.x], k0 = p.cu_k[it.x];
                    seq = make_int4(q0, p.cu_q[it.x + 1] - q0, p.cu_k[it.x + 1] - k0, k0);
                }
                s_item[slot][0] = it;
                s_item[slot][1] = itb;
                s_item[slot][2] = seq;
                mbar_arrive(item_full(slot));
                if (it.x < 0)
                    break;
                const int h = it.z;
                const ItemSpan sp = item_span(it, itb);
                if (sp.j1 <= sp.j0)
                    continue;
                for (int x = 0; x < 2 && ok; ++x) {
                    if (!sp.live(x))
                        continue;
                    const int i = x == 0 ? it.y : itb.x;
                    if (!mbar_wait(q_empty(x), (qloads[x] & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(q_full(x), C::Q_BYTES);
                    for (int db = 0; db < C::QK_DB; ++db)
                        tma_load_3d(sQ + x * C::Q_BYTES + db * (BQ * C::QK_ROW), &p.tm_q, q_full(x),
                                    db * C::QK_BLOCK, h, seq.x + i * BQ);
                    ++qloads[x];
                }
                for (int j = sp.j0; j < sp.j1 && ok; ++j) {
                    const int st = kfills % NS;
                    if (!mbar_wait(k_empty(st), ((kfills / NS) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full(st), C::K_BYTES);
                    for (int db = 0; db < C::QK_DB; ++db)
                        tma_load_3d(sK + st * C::K_BYTES + db * (BK * C::QK_ROW), &p.tm_k, k_full(st),
                                    db * C::QK_BLOCK, h / p.kv_group, seq.w + j * BK);
                    ++kfills;
                }
                if (!ok)
                    break;
            }
            if (!ok || *abort) {
                for (int st = 0; st < NS; ++st)
                    last_fill_wait(kfills, NS, st, k_full(st));
                for (int x = 0; x < 2; ++x)
                    if (qloads[x] > 0)
                        mbar_wait_drain(q_full(x), (qloads[x] - 1) & 1u);
            }
        }
    } else if (warp == kVWarp) {
        // ------------------------------------------------------------ V
        if (lane == 0) {
            uint32_t vfills = 0;
            bool ok = true;
            for (uint32_t n = 0;; ++n) {
                int4 it, itb, seq;
                const bool more = next_item(n, it, itb, seq);
                mbar_arrive(item_empty(n & 1));
                if (!more)
                    break;
                const int h = it.z;
                const ItemSpan sp = item_span(it, itb);
                for (int j = sp.j0; j < sp.j1; ++j) {
                    const int st = vfills % NS;
                    if (!mbar_wait(v_empty(st), ((vfills / NS) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full(st), C::KV_BYTES);
                    for (int db = 0; db < DB; ++db)
                        tma_load_3d(sV + st * C::KV_BYTES + db * (BK * 128), &p.tm_v, v_full(st),
                                    db * 64, h / p.kv_group, seq.w + j * BK);
                    ++vfills;
                }
                if (!ok)
                    break;
            }
            if (!ok || *abort)
                for (int st = 0; st < NS; ++st)
                    last_fill_wait(vfills, NS, st, v_full(st));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // All 32 lanes run this loop on warp-uniform values; one elected lane
        // issues each MMA and commit.
        {
            const uint64_t q_desc0 = C::QK_ROW == 128 ? sdesc_sw128(sQ, 16, 1024)
                                                      : sdesc_sw64(sQ, 16, 512);
            const uint64_t k_desc0 = C::QK_ROW == 128 ? sdesc_sw128(sK, 16, 1024)
                                                      : sdesc_sw64(sK, 16, 512);
            const uint64_t v_desc0 = sdesc_sw128(sV, BK * 128, 1024);
            uint32_t n = 0, kv = 0, qloads[2] = {0, 0}, gt[2] = {0, 0};   // tiles per q slot
            bool ok = true;
            // S_x = Q_x K^T for q slot x, K in ring slot st (issue order after the
            // previous O_x += P_x V protects P_x; see the file comment).
            auto issue_qk = [&](int x, int st) {
                const uint64_t qd = q_desc0 + x * (C::Q_BYTES >> 4);
                const uint64_t kd = k_desc0 + st * (C::K_BYTES >> 4);
                const uint32_t s_tm = tmem + C::S_COL + x * BK;
                // k-steps of 32 bytes: 16 bf16 or 32 FP8 elements
                // (KPB k-steps per swizzled row of QK_ROW bytes)
                constexpr int KPB = C::QK_ROW / 32;
#pragma unroll
                for (int kk = 0; kk < D / C::QK_KSTEP; ++kk) {
                    const uint64_t qo =
                        qd + (((kk / KPB) * (BQ * C::QK_ROW) + (kk % KPB) * 32) >> 4);
                    const uint64_t ko =
                        kd + (((kk / KPB) * (BK * C::QK_ROW) + (kk % KPB) * 32) >> 4);
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
            };
            // O_x += P_x V for q slot x (its tile number gt[x]), V in ring slot st,
            // one half of the keys as soon as the softmax has published that
            // half of P_x.
            auto issue_pv = [&](int x, int st, uint32_t v_fill, bool acc) -> bool {
                if (!mbar_wait(p_half(x, 0), gt[x] & 1u, abort) ||
                    !mbar_wait(v_full(st), (v_fill / NS) & 1u, abort))
                    return false;
                tc_fence_after();
                const uint64_t vd = v_desc0 + st * (C::KV_BYTES >> 4);
                const uint32_t a_tm = tmem + C::S_COL + x * BK;
                const uint32_t o_tm = tmem + x * D;
                if (acc)
                    mma_ts_w<1>(o_tm, a_tm, vd, C::IDESC_PV);
                else
                    mma_ts_w<0>(o_tm, a_tm, vd, C::IDESC_PV);
#pragma unroll
                for (int kk = 1; kk < BK / 32; ++kk)
                    mma_ts_w<1>(o_tm, a_tm + kk * 8, vd + kk * (16 * 128 / 16), C::IDESC_PV);
                mma_commit_w(o_h1(x));
                if (!mbar_wait(p_half(x, 1), gt[x] & 1u, abort))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int kk = BK / 32; kk < BK / 16; ++kk)
                    mma_ts_w<1>(o_tm, a_tm + kk * 8, vd + kk * (16 * 128 / 16), C::IDESC_PV);
                mma_commit_w(o_h2(x));
                ++gt[x];
                return true;
            };
            for (;; ++n) {
                int4 it, itb, seq;
                const bool more = next_item(n, it, itb, seq);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(item_empty(n & 1));
                if (!more)
                    break;
                const ItemSpan sp = item_span(it, itb);
                if (sp.j1 <= sp.j0)
                    continue;
                if ((sp.live(0) && !mbar_wait(q_full(0), qloads[0] & 1u, abort)) ||
                    (sp.live(1) && !mbar_wait(q_full(1), qloads[1] & 1u, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Slot x runs key tiles [first[x], end[x]) of the item's [j0, j1);
                // without a window both start at 0 and b's range ends first.
                for (int j = sp.j0; j < sp.j1 && ok; ++j) {
                    const int st = kv % NS;
                    const int st_prev = (kv + NS - 1) % NS;
                    const bool a_in = sp.has(0, j), b_in = sp.has(1, j);
                    if (!mbar_wait(k_full(st), (kv / NS) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    if (a_in) {
                        issue_qk(0, st);                          // S_a(j)
                        if (j == sp.end[0] - 1)
                            mma_commit_w(q_empty(0));
                    }
                    if (sp.has(1, j - 1)) {
                        // O_b += P_b(j-1) V(j-1); V(j-1) is then free
                        if (!issue_pv(1, st_prev, kv - 1, j - 1 > sp.first[1])) {
                            ok = false;
                            break;
                        }
                        mma_commit_w(v_empty(st_prev));
                    }
                    if (b_in) {
                        issue_qk(1, st);                          // S_b(j)
                        if (j == sp.end[1] - 1)
                            mma_commit_w(q_empty(1));
                    }
                    mma_commit_w(k_empty(st));
                    if (a_in && !issue_pv(0, st, kv, j > sp.first[0])) {   // O_a += P_a(j) V(j)
                        ok = false;
                        break;
                    }
                    if (!b_in) {
                        // tile b does not use V(j): free it now (after its fill
                        // has landed, if no product read it)
                        if (!a_in && !mbar_wait(v_full(st), (kv / NS) & 1u, abort)) {
                            ok = false;
                            break;
                        }
                        mma_commit_w(v_empty(st));
                    }
                    ++kv;
                }
                if (!ok)
                    break;
                if (sp.has(1, sp.j1 - 1)) {
                    const int st_last = (kv + NS - 1) % NS;
                    if (!issue_pv(1, st_last, kv - 1, sp.j1 - 1 > sp.first[1])) {
                        ok = false;
                        break;
                    }
                    mma_commit_w(v_empty(st_last));
                }
                if (sp.live(0))
                    ++qloads[0];
                if (sp.live(1))
                    ++qloads[1];
            }
            if (!ok || *abort) {
                mma_commit_w(drain_bar);
                mbar_wait_drain(drain_bar, 0);
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kMathRegs));
        // ------------------------------------------------------------ softmax / epilogue
        const int x = (warp - kFirstMathWarp) >> 2;   // q slot: 0 = tile a (warps 4-7), 1 = tile b
        const int quarter = warp & 3;                 // TMEM lanes [32*quarter, +32)
        const int r = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_addr + C::S_COL + x * BK;
        const uint32_t o_addr = tmem + lane_addr + x * D;
        const uint32_t wstage = sO + (warp - kFirstMathWarp) * C::WARP_STAGE;
        const float scale_log2 = p.scale_log2;
        const float2 scale2 = make_float2(scale_log2, scale_log2);
        const int H = p.num_heads;
        uint32_t g = 0;                               // this slot's tiles so far
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
        // Masked tiles mask the keys past a row's last visible one and, in the
        // sliding-window instantiation, those below the window's edge too (one
        // masked variant per instantiation keeps the register allocation of
        // the plain kernel).
        using Plain = std::integral_constant<int, 0>;
        using Masked = std::integral_constant<int, WIN ? 2 : 1>;

        for (uint32_t n = 0;; ++n) {
            int4 it, itb, seq;
            const bool more = next_item(n, it, itb, seq);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(item_empty(n & 1));
            if (!more)
                break;
            const int i = x == 0 ? it.y : itb.x;
            if (i < 0)
                continue;                             // no second tile in this item
            const int h = it.z;
            // this slot's key tiles [j_first, j_end)
            const int j_first = x == 0 ? itb.z : itb.w;
            const int j_end = x == 0 ? it.w : itb.y;
            const int q0 = seq.x, lq = seq.y, lk = seq.z;
            const int q_local = i * BQ + r;
            const bool row_valid = q_local < lq;
            const long long tok = static_cast<long long>(q0) + q_local;

            if (j_end <= j_first) {
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

            float m_used = -INFINITY;                 // reference max, log2 units
            float l = 0.f;
            bool ok = true;
            for (int j = j_first; j < j_end && ok; ++j) {
                if (!mbar_wait(s_full(x), g & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int k_base = j * BK;
                // causal: row q sees keys <= q + off (off = 0 top-left, Lk - Lq
                // bottom-right); a window also hides keys < q + off - window_left
                const int off = p.causal == 2 ? lk - lq : 0;
                const bool need_hi =
                    (k_base + BK > lk) || (p.causal && k_base + BK - 1 > i * BQ + off);
                // the tile's last row has the highest window edge
                const bool need_lo = WIN && k_base < static_cast<long long>(i) * BQ + BQ - 1 +
                                                         off - p.window_left;
                // this row's visible columns end at lim; warp-wide bounds of lim
                const bool need_mask = need_hi || need_lo;
                const int lim =
                    need_mask ? (p.causal ? min(lk, max(0, q_local + off + 1)) : lk) - k_base : BK;
                const int lim_lo = need_mask ? __reduce_min_sync(0xffffffffu, lim) : BK;
                const int lim_hi = need_mask ? __reduce_max_sync(0xffffffffu, lim) : BK;

                // The whole key tile's 128 scores of this row are loaded with one
                // wait.  The row max comes from the registers first; the reference
                // max moves (O, l rescaled) only if it grew by more than 2^8; then
                // p = 2^(s * scale_log2 - m) per 32-column chunk, stored as bf16
                // pairs over the chunk's first 16 S columns (all scores are in
                // registers by then), each half of P published on its own so that
                // O_x += P_x V starts on the first 64 keys while the second half is
                // being exponentiated.
                auto tile = [&](auto masked) -> bool {
                    constexpr int MK = decltype(masked)::value;
                    // banded tiles: this row's visible columns start at lo
                    int lo = 0, lo_lo = 0, lo_hi = 0;
                    if (MK == 2) {
                        const int off = p.causal == 2 ? lk - lq : 0;
                        lo = static_cast<int>(
                            min(static_cast<long long>(BK),
                                max(0ll, static_cast<long long>(q_local) + off - p.window_left -
                                             k_base)));
                        lo_lo = __reduce_min_sync(0xffffffffu, lo);
                        lo_hi = __reduce_max_sync(0xffffffffu, lo);
                    }
                    uint32_t sc[4][32];
                    tmem_ld32(s_addr, sc[0]);
                    tmem_ld32(s_addr + 32, sc[1]);
                    tmem_ld32(s_addr + 64, sc[2]);
                    tmem_ld32(s_addr + 96, sc[3]);
                    tmem_wait_ld_r(sc[0]);
                    tmem_bind_r(sc[1]);
                    tmem_bind_r(sc[2]);
                    tmem_bind_r(sc[3]);
                    // a chunk every row of the warp masks entirely
                    bool empty[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        empty[c] = MK > 0 && (32 * c >= lim_hi || (MK == 2 && 32 * c + 32 <= lo_lo));
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (empty[c])
                            continue;
                        if (MK > 0)
                            mask_chunk<MK == 2>(sc[c], 32 * c, lim, lim_lo, lo, lo_hi);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            mx[e & 3] = fmax3(mx[e & 3], __uint_as_float(sc[c][2 * e]),
                                              __uint_as_float(sc[c][2 * e + 1]));
                    }
                    const float mraw = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
                    const float m_tile = mraw == -INFINITY ? -INFINITY : mraw * scale_log2;
                    const float m_new = fmaxf(m_used, m_tile);
                    const bool grow = m_new > m_used + kRescaleThreshold;   // true for m_used = -inf
                    if (__any_sync(0xffffffffu, grow)) {
                        if (j > j_first) {
                            // O_x holds every product issued so far (the previous
                            // tile's, complete once S_x of this one is)
                            if (!mbar_wait(o_h2(x), (g - 1) & 1u, abort))
                                return false;
                            tc_fence_after();
                            const float f = grow ? ex2_approx(m_used - m_new) : 1.f;
                            rescale_rows<D>(o_addr, f);
                            l *= f;
                        }
                        if (grow)
                            m_used = m_new;
                    }
                    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
                    const float2 negm2 = make_float2(neg_m, neg_m);
                    float2 ls[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        ls[e] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
                        if (empty[c]) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                pk[e] = 0u;
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 t = __ffma2_rn(
                                    make_float2(__uint_as_float(sc[c][2 * e]),
                                                __uint_as_float(sc[c][2 * e + 1])),
                                    scale2, negm2);
                                const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                                ls[e & 3] = __fadd2_rn(ls[e & 3], pp);
                                pk[e] = pack_bf16x2(pp.x, pp.y);
                            }
                        }
                        tmem_st16(s_addr + 16 * c, pk);
                        if (c & 1) {
                            tmem_wait_st();
                            tc_fence_before();
                            mbar_arrive(p_half(x, c >> 1));
                        }
                    }
                    const float2 l2 = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
                    l += l2.x + l2.y;
                    return true;
                };
                ok = need_mask ? tile(Masked{}) : tile(Plain{});
                ++g;
            }
            if (!ok)
                break;

            // Epilogue: wait for this tile's last O += P V, then O / l -> bf16 and lse.
            if (!mbar_wait(o_h2(x), (g - 1) & 1u, abort))
                break;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            if (row_valid)
                p.lse[tok * H + h] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -FLT_MAX;
            // O / l -> bf16, 32 columns at a time through this warp's stage: each
            // thread writes its row segment (swizzled as the 64-byte TMA swizzle
            // lays it out, conflict-free).  A warp whose 32 rows all belong to the
            // sequence then hands the chunk to a TMA tile store; otherwise (the
            // sequence's last tile: rows past it belong to the next sequence)
            // every store instruction writes eight whole 64-byte row segments of
            // the rows that exist.
            const int tile_rows = min(BQ, lq - i * BQ);
            const bool warp_rows = quarter * 32 + 32 <= tile_rows;   // warp-uniform
            __nv_bfloat16 *out_tile = out + ((static_cast<long long>(q0) + i * BQ) * H + h) * D;
#pragma unroll
            for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t rr[32];
                tmem_ld32(o_addr + cb * 32, rr);
                tmem_wait_ld_r(rr);
                // the stage's previous tile store has read it
                if (lane == 0)
                    bulk_wait_group_read0();
                __syncwarp();
                const uint32_t row = wstage + lane * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(row + ((c ^ ((lane >> 1) & 3)) << 4),
                                 pack_bf16x2(__uint_as_float(rr[8 * c + 0]) * inv_l,
                                             __uint_as_float(rr[8 * c + 1]) * inv_l),
                                 pack_bf16x2(__uint_as_float(rr[8 * c + 2]) * inv_l,
                                             __uint_as_float(rr[8 * c + 3]) * inv_l),
                                 pack_bf16x2(__uint_as_float(rr[8 * c + 4]) * inv_l,
                                             __uint_as_float(rr[8 * c + 5]) * inv_l),
                                 pack_bf16x2(__uint_as_float(rr[8 * c + 6]) * inv_l,
                                             __uint_as_float(rr[8 * c + 7]) * inv_l));
                if (warp_rows) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&p.tm_o, wstage, cb * 32, h, q0 + i * BQ + quarter * 32);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rw = 8 * k + (lane >> 2), ch = lane & 3;
                        const int rt = quarter * 32 + rw;          // row within the tile
                        const uint4 v =
                            ld_shared_v4(wstage + rw * 64 + ((ch ^ ((rw >> 1) & 3)) << 4));
                        if (rt < tile_rows)
                            *reinterpret_cast<uint4 *>(out_tile + static_cast<long long>(rt) * H * D +
                                                       cb * 32 + ch * 8) = v;
                    }
                    __syncwarp();
                }
            }
        }
        // every tile store of this warp has completed before the CTA exits
        if (lane == 0)
            bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 0)
        atomicCAS(p.status, 0, VFA_ERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool WIN, bool F8>
cudaError_t launch_pair_dw(const PrefillArgs &a, int grid, cudaStream_t stream)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(prefill_pair_kernel<D, WIN, F8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PairCfg<D, F8>::SMEM));
        if (e != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PairCfg<D, F8>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel<D, WIN, F8>, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// The sliding-window mask and FP8 Q / K have their own instantiations.
template <int D>
cudaError_t launch_pair_d(const PrefillArgs &a, int grid, cudaStream_t stream)
{
    if (a.qk_fp8)
        return a.window_left >= 0 ? launch_pair_dw<D, true, true>(a, grid, stream)
                                  : launch_pair_dw<D, false, true>(a, grid, stream);
    return a.window_left >= 0 ? launch_pair_dw<D, true, false>(a, grid, stream)
                              : launch_pair_dw<D, false, false>(a, grid, stream);
}

}  // namespace

cudaError_t launch_prefill_pair(int head_dim, const PrefillArgs &a, int grid, cudaStream_t stream)
{
    switch (head_dim) {
    case 64: return launch_pair_d<64>(a, grid, stream);
    case 128: return launch_pair_d<128>(a, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vfa
