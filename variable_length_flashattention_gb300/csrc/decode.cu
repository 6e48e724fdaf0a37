// decode.cu -- paged GQA decode on sm_103a: state init, one tile step, finalize.
//
// Follows "attention_ref.rs" (spark_storage): AttnState::new (m = -inf,
// l = 0, o = 0), step_tile_ref (every block_size token of every listed block
// updates the running max, denominator and weighted V sum of each q head,
// logits (q . k) / sqrt(D), kv head = q head / group) and finalize_ref
// (o / l, 0 when l = 0, rounded to bf16).  The reference walks tokens one by
// one; here the work is memory-bound and laid out for HBM:
//
//   * one CTA per (kv head, sequence): the group of q heads that share a kv
//     head is handled together, so each K/V block row is read from HBM once;
//   * the listed blocks stream by TMA through a ring of shared-memory stages
//     (48 KB per CTA), each of the CTA's four warps computing on every fourth
//     block, so HBM reads for later blocks overlap the arithmetic on earlier
//     ones, and four CTAs fit on an SM: all (kv head, sequence) CTAs of a
//     64-sequence, 8-kv-head batch are resident at once;
//   * per block, S = K Q^T and O^T += V^T P run on the warp-level tensor
//     instruction (mma.sync, bf16 in, fp32 accumulate; q heads padded to 8):
//     the kernel stays bound by HBM, and these 16-token products would cost
//     an order of magnitude more instructions as scalar FMAs;
//   * the warps' partial states are merged in shared memory with the
//     incoming state, all relative to one max, and written back (m in
//     natural-log units).
// Block ids and counts are validated before any state is touched; bad ones
// set VFA_ERR_BAD_BLOCK and leave that sequence's state as it was.
#include <cfloat>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace vfa {

namespace {

constexpr int kWarps = 4;
constexpr int kBlockSize = 16;          // tokens per KV block (the supported size)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;


// Row of kv head `kh`, token `t` of physical block `blk` in a
// [num_blocks, block_size, num_kv_heads, D] pool: the one address rule of
// both the step kernel and the gather test hook.
template <int D>
__device__ __forceinline__ const __nv_bfloat16 *kv_row(const void *pool, int blk, int t, int kh,
                                                        int num_kv_heads)
{
    const long long row = (static_cast<long long>(blk) * kBlockSize + t) * num_kv_heads + kh;
    return static_cast<const __nv_bfloat16 *>(pool) + row * D;
}

// This lane's DPL = D/16 consecutive elements of a row, as DPL/2 bf16x2 words.
template <int D>
__device__ __forceinline__ void load_chunk(const __nv_bfloat16 *row, int l16, uint32_t *w)
{
    constexpr int DPL = D / 16;
    const __nv_bfloat16 *src = row + l16 * DPL;
    if constexpr (DPL == 4) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(src));
        w[0] = v.x; w[1] = v.y;
    } else if constexpr (DPL == 8) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(src));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
        const uint4 v0 = __ldcs(reinterpret_cast<const uint4 *>(src));
        const uint4 v1 = __ldcs(reinterpret_cast<const uint4 *>(src) + 1);
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    }
}

// Waits (bounded, like mbar_wait) until the shared counter *c exceeds n.
__device__ __forceinline__ bool wait_count_above(const int *c, int n, volatile int *abort)
{
    const volatile int *vc = c;
    if (*vc > n)
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (*vc > n)
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// Validates tile_blocks[s, 0:count] and the count; every thread of the CTA
// gets the same verdict.
__device__ __forceinline__ bool tile_row_valid(const int32_t *tile_blocks, int count, int cap,
                                               int num_blocks, int s)
{
    bool bad = (count < 0 || count > cap);
    if (!bad) {
        for (int b = threadIdx.x; b < count; b += blockDim.x) {
            const int blk = tile_blocks[static_cast<long long>(s) * cap + b];
            bad |= (blk < 0 || blk >= num_blocks);
        }
    }
    return !__syncthreads_or(bad);
}

// ------------------------------------------------------------ step kernel
//
// One CTA of kStepWarps warps per (kv head, sequence).  The tile's blocks
// stream through one ring of NS shared-memory stages: block k goes to stage
// k % NS by TMA (K and V of one block for this kv head are D/64 boxes of 16
// tokens x 64 columns each, 128-byte swizzled, from the pool viewed as
// [blocks * 16 tokens, kv heads, D]); warp k % 4 consumes it and then
// refills the stage with block k + NS, so up to NS blocks are in flight
// while the warps compute.
//
// A warp's work on one block is two thin products on the warp-level tensor
// instruction (mma.sync m16n8k16, bf16 in, fp32 accumulate), which keeps the
// instruction count per byte low enough for HBM to be the limit:
//   S[16 tokens x 8]   = K[16 x D] . Q^T[D x 8]       (q heads padded to 8)
//   O^T[D x 8]        += V^T[D x 16] . P[16 tokens x 8]
// K comes in with ldmatrix, V^T with ldmatrix.trans; P leaves S's fragment
// transposed by movmatrix.  In both accumulators a lane holds heads
// 2*(lane % 4) and 2*(lane % 4) + 1, so the running max, the rescale of O
// and p need no exchange beyond a max over the 8 lanes sharing those heads.
constexpr int kStepWarps = 4;
constexpr int kRingBytes = 48 * 1024;

template <int D>
struct StepCfg {
    static constexpr int STAGE = 2 * kBlockSize * D * 2;         // K and V of one block
    static constexpr int NS = kRingBytes / STAGE;                 // 12, 6, 3 stages
    static constexpr int RING = NS * STAGE;
    static constexpr int KB = D / 64;                             // 64-column boxes per row
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// c[0..3] += A(16x16, a[0..3]) * B(16x8, b[0..1]), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared address of the 16-byte chunk `chunk` (8 columns) of token row `row`
// in one 16-row operand of D/64 swizzled 64-column boxes (2 KB each).
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int row, int chunk)
{
    return base + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// SPLIT: the CTA takes run blockIdx.z of the tile's blocks (the split step)
// and merges through the workspace instead of into the state directly.
template <int D, int G, bool SPLIT>
__global__ void __launch_bounds__(kStepWarps * 32) decode_step_kernel(
    const DecodeStepArgs a, const __grid_constant__ DecodeMaps t)
{
    using C = StepCfg<D>;
    constexpr int NS = C::NS;
    constexpr int MT = D / 16;                // 16-column tiles of D

    extern __shared__ __align__(1024) uint8_t dsm_raw[];
    // 128-byte swizzled TMA destinations start on a 1024-byte boundary.
    uint8_t *dsm = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(dsm + C::RING);            // [NS]
    __shared__ float s_m[kStepWarps][8], s_l[kStepWarps][8];
    __shared__ float s_min[G], s_lin[G];
    __shared__ int s_abort;
    __shared__ int s_fills[NS], s_used[NS];   // per stage: fills issued, fills consumed
    __shared__ int s_last;

    const int kh = blockIdx.x;
    const int s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = a.num_q_heads;

    // Consecutive steps are launched with programmatic serialisation: the
    // next step may start streaming its blocks now; it waits for this grid
    // (griddepcontrol.wait) before it touches the state or the status word.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int count = a.tile_block_counts[s];
    // Tokens to absorb: the first n_tok of the listed blocks' tokens.
    const int n_tok = a.tile_token_counts ? a.tile_token_counts[s]
                      : (count >= 0 && count <= a.tile_capacity ? count * kBlockSize : 0);
    const bool tok_bad = n_tok < 0 || static_cast<long long>(n_tok) >
                                          static_cast<long long>(count) * kBlockSize;
    if (!tile_row_valid(a.tile_blocks, count, a.tile_capacity, a.num_blocks, s) || tok_bad) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (threadIdx.x == 0 && a.status)
            atomicCAS(a.status, 0, VFA_ERR_BAD_BLOCK);
        return;
    }
    if (count == 0 || n_tok == 0)
        return;                                 // an empty tile leaves the state as it was
    const int nb_all = (n_tok + kBlockSize - 1) / kBlockSize;   // blocks holding those tokens
    // This CTA's run of blocks [kb0, kb0 + nb): the whole tile, or run
    // blockIdx.z of num_splits equal runs (possibly empty).
    int kb0 = 0, nb = nb_all;
    if (SPLIT) {
        const int per = (nb_all + a.num_splits - 1) / a.num_splits;
        kb0 = min(nb_all, static_cast<int>(blockIdx.z) * per);
        nb = min(nb_all, kb0 + per) - kb0;
    }

    const uint32_t ring = smem_u32(dsm);
    auto stage_k = [&](int st) { return ring + st * C::STAGE; };
    auto full = [&](int st) { return smem_u32(&bars[st]); };
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            s_fills[i] = 0;
            s_used[i] = 0;
        }
        fence_barrier_init();
    }
    __syncthreads();
    volatile int *abort = &s_abort;

    const int32_t *row_ids = a.tile_blocks + static_cast<long long>(s) * a.tile_capacity + kb0;
    // Block k of the run into stage k % NS (one thread issues a fill).
    auto issue = [&](int k) {
        const int blk = row_ids[k];
        const int st = k % NS;
        mbar_arrive_expect_tx(full(st), C::STAGE);
#pragma unroll
        for (int b = 0; b < C::KB; ++b) {
            tma_load_3d(stage_k(st) + b * 2048, &t.tm_k, full(st), b * 64, kh, blk * kBlockSize);
            tma_load_3d(stage_k(st) + C::STAGE / 2 + b * 2048, &t.tm_v, full(st), b * 64, kh,
                        blk * kBlockSize);
        }
        // Published after the arrive: a consumer that sees the new count waits
        // on a barrier already armed for this fill.
        __threadfence_block();
        atomicAdd(&s_fills[st], 1);
    };
    if (threadIdx.x == 0)
        for (int k = 0; k < NS && k < nb; ++k)
            issue(k);

    // Q^T fragments (B operand of S = K Q^T): head n = lane / 4, columns
    // 16 * kt + 2 * (lane % 4) + {0, 1} and + 8; heads past G are zero.
    const int n_q = lane >> 2, t4 = lane & 3;
    uint32_t qb[MT][2];
    {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            static_cast<const __nv_bfloat16 *>(a.q) +
            (static_cast<long long>(s) * Hq + kh * G + (n_q < G ? n_q : 0)) * D);
#pragma unroll
        for (int kt = 0; kt < MT; ++kt) {
            qb[kt][0] = n_q < G ? qrow[(16 * kt + 2 * t4) / 2] : 0u;
            qb[kt][1] = n_q < G ? qrow[(16 * kt + 8 + 2 * t4) / 2] : 0u;
        }
    }
    const float sc = a.scale_log2;                            // logits in log2 units

    // This lane's two heads: 2 * t4 and 2 * t4 + 1.
    float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[mt][e] = 0.f;
    // ldmatrix row addresses: lane L serves row L % 8 of 8x8 matrix L / 8.
    const int mi = lane >> 3, mr = lane & 7;
    const int k_row = ((mi & 1) << 3) + mr, k_chunk = mi >> 1;     // K: A of S = K Q^T
    const int v_row = ((mi >> 1) << 3) + mr, v_chunk = mi & 1;     // V^T: A of O^T += V^T P

    for (int k = warp; k < nb; k += kStepWarps) {
        const int st = k % NS;
        const int fill = k / NS;
        // The parity wait below is only unambiguous once this stage's previous
        // fill has completed, and another warp may get here first: wait until
        // this fill has been issued (its issuer consumed the previous one).
        if (!wait_count_above(&s_fills[st], fill, abort) ||
            !mbar_wait(full(st), fill & 1u, abort))
            break;
        const uint32_t sk = stage_k(st), sv = sk + C::STAGE / 2;

        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < MT; ++kt) {
            uint32_t af[4];
            ldsm_x4(sw_addr(sk, k_row, 2 * kt + k_chunk), af);
            mma_bf16(sacc, af, qb[kt][0], qb[kt][1]);
        }
        // sacc: tokens lane/4 (0, 1) and lane/4 + 8 (2, 3); heads 2*t4 (0, 2), 2*t4+1 (1, 3).
        // Tokens past n_tok (only in the last block) get weight zero; every
        // block read holds at least one token that counts.
        const int valid = n_tok - (kb0 + k) * kBlockSize;
        if (valid < kBlockSize) {
            const int t0 = lane >> 2;
            if (t0 >= valid) {
                sacc[0] = -INFINITY;
                sacc[1] = -INFINITY;
            }
            if (t0 + 8 >= valid) {
                sacc[2] = -INFINITY;
                sacc[3] = -INFINITY;
            }
        }
        float bm[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float x = fmaxf(sacc[h], sacc[h + 2]) * sc;
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1)
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
            bm[h] = x;
        }
        float f[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mnew = fmaxf(m_run[h], bm[h]);
            f[h] = ex2_approx(m_run[h] - mnew);            // 0 when m_run = -inf, 1 if unchanged
            m_run[h] = mnew;
            l_part[h] *= f[h];
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            o[mt][0] *= f[0];
            o[mt][1] *= f[1];
            o[mt][2] *= f[0];
            o[mt][3] *= f[1];
        }
        const float p0 = ex2_approx(sacc[0] * sc - m_run[0]);
        const float p1 = ex2_approx(sacc[1] * sc - m_run[1]);
        const float p2 = ex2_approx(sacc[2] * sc - m_run[0]);
        const float p3 = ex2_approx(sacc[3] * sc - m_run[1]);
        l_part[0] += p0 + p2;
        l_part[1] += p1 + p3;
        // P as two 8x8 tiles (tokens 0-7, 8-15) x 8 heads, transposed into the
        // B operand (k = token, n = head) of O^T += V^T P.
        const uint32_t pb0 = movm_t(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movm_t(pack_bf16x2(p2, p3));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t af[4];
            ldsm_x4_t(sw_addr(sv, v_row, 2 * mt + v_chunk), af);
            mma_bf16(o[mt], af, pb0, pb1);
        }
        // Every lane is done with this stage: refill it with block k + NS.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            ++s_used[st];
            if (k + NS < nb)
                issue(k + NS);
        }
    }
    // Warp totals of l: the 8 lanes sharing this lane's heads (lane % 4).
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float x = l_part[h];
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1)
            x += __shfl_xor_sync(0xffffffffu, x, off);
        l_part[h] = x;
    }
    __syncthreads();                                    // every warp is out of the ring
    // The previous step (or the init) must be complete before its state is
    // read, and (split step) before the shared workspace is written.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!SPLIT && *abort) {
        // A stage's last fill may still be in flight if nobody consumed it:
        // wait for it (bounded) before the CTA exits; the state is left as it was.
        if (threadIdx.x == 0) {
            for (int st = 0; st < NS; ++st)
                if (s_fills[st] > s_used[st])
                    mbar_wait_drain(full(st), (s_fills[st] - 1) & 1u);
            if (a.status)
                atomicCAS(a.status, 0, VFA_ERR_TIMEOUT);
        }
        return;
    }
    if (SPLIT && *abort) {
        // the partial is not usable: contribute an empty one, keep the tickets whole
        if (threadIdx.x == 0)
            for (int st = 0; st < NS; ++st)
                if (s_fills[st] > s_used[st])
                    mbar_wait_drain(full(st), (s_fills[st] - 1) & 1u);
        __syncthreads();
        if (lane < 4)
            for (int h = 0; h < 2; ++h) {
                m_run[h] = -INFINITY;
                l_part[h] = 0.f;
            }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[mt][e] = 0.f;
        if (threadIdx.x == 0 && a.status)
            atomicCAS(a.status, 0, VFA_ERR_TIMEOUT);
    }
    float *s_o = reinterpret_cast<float *>(dsm);        // [warps][G][D], over the ring
    if (lane < 4) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            s_m[warp][2 * lane + h] = m_run[h];
            s_l[warp][2 * lane + h] = l_part[h];
        }
    }
    // o[mt]: columns 16*mt + lane/4 (0, 1) and + 8 (2, 3); heads 2*t4 (0, 2), 2*t4+1 (1, 3).
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = 2 * t4 + (e & 1);
            const int col = 16 * mt + (lane >> 2) + ((e >> 1) << 3);
            if (h < G)
                s_o[(warp * G + h) * D + col] = o[mt][e];
        }
    if (SPLIT) {
        // This CTA's partial state, its warps merged relative to one max
        // (log2 units): [g][0] = m, [g][1] = l, [g][2 ..] = o.
        __syncthreads();
        const int row = s * a.num_kv_heads + kh;
        float *part = a.part + (static_cast<long long>(row) * a.num_splits + blockIdx.z) * G *
                                   (D + 2);
        for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
            const int g = e / D, d = e % D;
            float mt = s_m[0][g];
#pragma unroll
            for (int w = 1; w < kStepWarps; ++w)
                mt = fmaxf(mt, s_m[w][g]);
            float acc_o = 0.f, acc_l = 0.f;
            if (mt != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kStepWarps; ++w) {
                    const float fw = ex2_approx(s_m[w][g] - mt);
                    acc_o = fmaf(s_o[(w * G + g) * D + d], fw, acc_o);
                    acc_l = fmaf(s_l[w][g], fw, acc_l);
                }
            }
            part[g * (D + 2) + 2 + d] = acc_o;
            if (d == 0) {
                part[g * (D + 2)] = mt;
                part[g * (D + 2) + 1] = acc_l;
            }
        }
        // Publish the partial, then take a ticket; the last CTA of the row merges.
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0)
            s_last = atomicAdd(a.tickets + row, 1) == a.num_splits - 1;
        __syncthreads();
        if (!s_last)
            return;
        __threadfence();
        const float *parts = a.part + static_cast<long long>(row) * a.num_splits * G * (D + 2);
        // per head: the merged max and the weights of the incoming state (w[0])
        // and of each run (w[1 + c]), over the ring, which is free now
        const int NW = a.num_splits + 1;
        float *s_w = reinterpret_cast<float *>(dsm);          // [G][NW]
        __syncthreads();
        if (threadIdx.x < G) {
            const int g = threadIdx.x;
            const long long sh = static_cast<long long>(s) * Hq + kh * G + g;
            const float m_in = a.m[sh] * kLog2e;
            float mt = m_in;
            for (int c = 0; c < a.num_splits; ++c)
                mt = fmaxf(mt, __ldcg(parts + (c * G + g) * (D + 2)));
            const bool live = mt != -INFINITY;
            s_w[g * NW] = live ? ex2_approx(m_in - mt) : 0.f;   // 0 for a fresh state
            for (int c = 0; c < a.num_splits; ++c)
                s_w[g * NW + 1 + c] =
                    live ? ex2_approx(__ldcg(parts + (c * G + g) * (D + 2)) - mt) : 0.f;
            s_min[g] = mt;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
            const int g = e / D, d = e % D;
            const long long sh = static_cast<long long>(s) * Hq + kh * G + g;
            const float *w = s_w + g * NW;
            float acc_o = a.o[sh * D + d] * w[0];
            for (int c = 0; c < a.num_splits; ++c)
                acc_o = fmaf(__ldcg(parts + (c * G + g) * (D + 2) + 2 + d), w[1 + c], acc_o);
            a.o[sh * D + d] = acc_o;
            if (d == 0) {
                float acc_l = a.l[sh] * w[0];
                for (int c = 0; c < a.num_splits; ++c)
                    acc_l = fmaf(__ldcg(parts + (c * G + g) * (D + 2) + 1), w[1 + c], acc_l);
                a.l[sh] = acc_l;
                a.m[sh] = s_min[g] == -INFINITY ? -INFINITY : s_min[g] * kLn2;
            }
        }
        if (threadIdx.x == 0)
            a.tickets[row] = 0;                          // ready for the next call
        return;
    }
    if (threadIdx.x < G) {
        const long long sh = static_cast<long long>(s) * Hq + kh * G + threadIdx.x;
        s_min[threadIdx.x] = a.m[sh] * kLog2e;
        s_lin[threadIdx.x] = a.l[sh];
    }
    __syncthreads();

    // Merge the warps with the incoming state (stored m is in natural-log units).
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
        const int g = e / D, d = e % D;
        const long long sh = static_cast<long long>(s) * Hq + kh * G + g;
        const float m_in = s_min[g];
        float mt = m_in;
#pragma unroll
        for (int w = 0; w < kStepWarps; ++w)
            mt = fmaxf(mt, s_m[w][g]);
        const float f_in = ex2_approx(m_in - mt);      // 0 for a fresh state (m_in = -inf)
        float acc_o = a.o[sh * D + d] * f_in;
        float acc_l = s_lin[g] * f_in;
#pragma unroll
        for (int w = 0; w < kStepWarps; ++w) {
            const float fw = ex2_approx(s_m[w][g] - mt);   // 0 for a warp with no blocks
            acc_o = fmaf(s_o[(w * G + g) * D + d], fw, acc_o);
            acc_l = fmaf(s_l[w][g], fw, acc_l);
        }
        a.o[sh * D + d] = acc_o;
        if (d == 0) {
            a.l[sh] = acc_l;
            a.m[sh] = mt * kLn2;
        }
    }
}

template <int D, int G>
size_t step_smem_bytes()
{
    return 1024 + StepCfg<D>::RING + StepCfg<D>::NS * sizeof(uint64_t);
}

__global__ void decode_init_kernel(float *m, float *l, float *o, long long n_state, int head_dim,
                                   int32_t *status)
{
    // A following step may launch now; it waits for this grid before it
    // reads the state.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         i < n_state * head_dim; i += stride) {
        o[i] = 0.f;
        if (i < n_state) {
            m[i] = -INFINITY;
            l[i] = 0.f;
        }
    }
    if (status && blockIdx.x == 0 && threadIdx.x == 0)
        *status = VFA_OK;
}

// out = bf16(o * (l > 0 ? 1/l : 0)), eight elements per thread.
__global__ void decode_finalize_kernel(const float *l, const float *o, long long n_state,
                                       int head_dim, __nv_bfloat16 *out)
{
    const long long n8 = n_state * head_dim / 8;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
         i += stride) {
        const long long e0 = i * 8;
        const float lv = l[e0 / head_dim];
        const float inv = lv > 0.f ? 1.f / lv : 0.f;
        const float4 a = reinterpret_cast<const float4 *>(o)[2 * i];
        const float4 b = reinterpret_cast<const float4 *>(o)[2 * i + 1];
        uint4 r;
        r.x = pack_bf16x2(a.x * inv, a.y * inv);
        r.y = pack_bf16x2(a.z * inv, a.w * inv);
        r.z = pack_bf16x2(b.x * inv, b.y * inv);
        r.w = pack_bf16x2(b.z * inv, b.w * inv);
        reinterpret_cast<uint4 *>(out)[i] = r;
    }
}

// Test hook: the step kernel's gather, written out instead of consumed.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) decode_gather_kernel(const DecodeStepArgs a,
                                                                     __nv_bfloat16 *k_out,
                                                                     __nv_bfloat16 *v_out)
{
    constexpr int DPL = D / 16, W = DPL / 2, TPL = kBlockSize / 2;
    const int kh = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int Hkv = a.num_kv_heads;
    const int count = a.tile_block_counts[s];
    if (!tile_row_valid(a.tile_blocks, count, a.tile_capacity, a.num_blocks, s)) {
        if (threadIdx.x == 0 && a.status)
            atomicCAS(a.status, 0, VFA_ERR_BAD_BLOCK);
        return;
    }
    const int32_t *row_ids = a.tile_blocks + static_cast<long long>(s) * a.tile_capacity;
    for (int bi = warp; bi < count; bi += kWarps) {
        const int blk = row_ids[bi];
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
            const int t = 2 * i + half;
            uint32_t kw[W], vw[W];
            load_chunk<D>(kv_row<D>(a.k_pool, blk, t, kh, Hkv), l16, kw);
            load_chunk<D>(kv_row<D>(a.v_pool, blk, t, kh, Hkv), l16, vw);
            const long long dst =
                (((static_cast<long long>(s) * a.tile_capacity + bi) * kBlockSize + t) * Hkv + kh) * D +
                l16 * DPL;
            uint32_t *kd = reinterpret_cast<uint32_t *>(k_out + dst);
            uint32_t *vd = reinterpret_cast<uint32_t *>(v_out + dst);
#pragma unroll
            for (int e = 0; e < W; ++e) {
                kd[e] = kw[e];
                vd[e] = vw[e];
            }
        }
    }
}

template <int D, int G, bool SPLIT>
cudaError_t step_dgs(const DecodeStepArgs &a, const DecodeMaps &maps, cudaStream_t stream)
{
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const size_t smem = step_smem_bytes<D, G>();
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_step_kernel<D, G, SPLIT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        attr_done[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_kv_heads, a.num_seqs, SPLIT ? a.num_splits : 1);
    cfg.blockDim = dim3(kStepWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_step_kernel<D, G, SPLIT>, a, maps);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t step_dg(const DecodeStepArgs &a, const DecodeMaps &maps, cudaStream_t stream)
{
    return a.num_splits > 1 ? step_dgs<D, G, true>(a, maps, stream)
                            : step_dgs<D, G, false>(a, maps, stream);
}

template <int D>
cudaError_t step_d(const DecodeStepArgs &a, const DecodeMaps &maps, cudaStream_t stream)
{
    switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return step_dg<D, 1>(a, maps, stream);
    case 2: return step_dg<D, 2>(a, maps, stream);
    case 4: return step_dg<D, 4>(a, maps, stream);
    case 8: return step_dg<D, 8>(a, maps, stream);
    default: return cudaErrorInvalidValue;
    }
}

int grid_for(long long n, int threads)
{
    long long g = (n + threads - 1) / threads;
    if (g < 1)
        g = 1;
    if (g > 4096)
        g = 4096;
    return static_cast<int>(g);
}

}  // namespace

size_t decode_split_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int num_splits)
{
    size_t n = static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(int32_t);   // tickets
    n = (n + 255) & ~static_cast<size_t>(255);
    n += static_cast<size_t>(num_seqs) * num_q_heads * num_splits * (head_dim + 2) *
         sizeof(float);
    return (n + 255) & ~static_cast<size_t>(255);
}

void decode_split_workspace_carve(void *ws, int num_seqs, int num_kv_heads, DecodeStepArgs *a)
{
    uint8_t *p = static_cast<uint8_t *>(ws);
    a->tickets = reinterpret_cast<int32_t *>(p);
    size_t n = static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(int32_t);
    n = (n + 255) & ~static_cast<size_t>(255);
    a->part = reinterpret_cast<float *>(p + n);
}

cudaError_t launch_decode_init(float *m, float *l, float *o, int num_seqs, int num_q_heads,
                               int head_dim, int32_t *status, cudaStream_t stream)
{
    const long long n_state = static_cast<long long>(num_seqs) * num_q_heads;
    decode_init_kernel<<<grid_for(n_state * head_dim, 256), 256, 0, stream>>>(m, l, o, n_state,
                                                                             head_dim, status);
    return cudaGetLastError();
}

cudaError_t launch_decode_step(const DecodeStepArgs &a, const DecodeMaps &maps,
                               cudaStream_t stream)
{
    switch (a.head_dim) {
    case 64: return step_d<64>(a, maps, stream);
    case 128: return step_d<128>(a, maps, stream);
    case 256: return step_d<256>(a, maps, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_finalize(const float *l, const float *o, int num_seqs, int num_q_heads,
                                   int head_dim, void *out, cudaStream_t stream)
{
    const long long n_state = static_cast<long long>(num_seqs) * num_q_heads;
    decode_finalize_kernel<<<grid_for(n_state * head_dim / 8, 256), 256, 0, stream>>>(
        l, o, n_state, head_dim, static_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError();
}

cudaError_t launch_decode_gather(const DecodeStepArgs &a, void *k_out, void *v_out,
                                 cudaStream_t stream)
{
    dim3 grid(a.num_kv_heads, a.num_seqs);
    auto *ko = static_cast<__nv_bfloat16 *>(k_out);
    auto *vo = static_cast<__nv_bfloat16 *>(v_out);
    switch (a.head_dim) {
    case 64: decode_gather_kernel<64><<<grid, kWarps * 32, 0, stream>>>(a, ko, vo); break;
    case 128: decode_gather_kernel<128><<<grid, kWarps * 32, 0, stream>>>(a, ko, vo); break;
    case 256: decode_gather_kernel<256><<<grid, kWarps * 32, 0, stream>>>(a, ko, vo); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace vfa
