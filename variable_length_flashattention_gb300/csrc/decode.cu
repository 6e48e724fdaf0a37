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
//   * each warp takes every 4th listed block; a block is 16 tokens x D,
//     read with 16-byte vector loads (16 lanes per token row, two tokens per
//     warp-wide load); fp32 FMA dot products, no tensor cores (the
//     contraction is 16 tokens by a handful of heads, far too thin);
//   * per block, the 16-lane partial dot products are reduced by a transposing
//     butterfly (each level halves the values a lane holds), the block max
//     and exponentials follow, and the block's p values are broadcast back to
//     the lanes that own V's columns;
//   * the four warps' partial states are merged in shared memory with the
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

// bf16x2 word -> two floats (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

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

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32) decode_step_kernel(const DecodeStepArgs a)
{
    constexpr int DPL = D / 16;             // elements per lane per token row
    constexpr int W = DPL / 2;              // bf16x2 words per lane per row
    constexpr int TPL = kBlockSize / 2;     // tokens per lane per block (two per warp load)
    constexpr int NV = TPL * G;             // partial dot products per lane before reduction
    constexpr int KPL = G >= 2 ? G / 2 : 1; // complete dot products per lane after reduction

    __shared__ float s_m[kWarps][G];
    __shared__ float s_l[kWarps][G];
    __shared__ float s_o[kWarps][G][D];

    const int kh = blockIdx.x;
    const int s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;

    const int count = a.tile_block_counts[s];
    if (!tile_row_valid(a.tile_blocks, count, a.tile_capacity, a.num_blocks, s)) {
        if (threadIdx.x == 0 && a.status)
            atomicCAS(a.status, 0, VFA_ERR_BAD_BLOCK);
        return;
    }
    if (count == 0)
        return;                                 // an empty tile leaves the state as it was

    // q of the G heads of this group, pre-scaled by log2(e)/sqrt(D): this lane's columns.
    const float qscale = kLog2e * rsqrtf(static_cast<float>(D));
    float qv[G][DPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16 *qrow =
            static_cast<const __nv_bfloat16 *>(a.q) + (static_cast<long long>(s) * Hq + kh * G + g) * D;
        uint32_t w[W];
        const uint32_t *src = reinterpret_cast<const uint32_t *>(qrow + l16 * DPL);
#pragma unroll
        for (int e = 0; e < W; ++e)
            w[e] = src[e];
#pragma unroll
        for (int e = 0; e < W; ++e) {
            qv[g][2 * e] = bf_lo(w[e]) * qscale;
            qv[g][2 * e + 1] = bf_hi(w[e]) * qscale;
        }
    }

    float m_run[G], l_part[G], o[G][DPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_part[g] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d)
            o[g][d] = 0.f;
    }

    const int32_t *row_ids = a.tile_blocks + static_cast<long long>(s) * a.tile_capacity;
    for (int bi = warp; bi < count; bi += kWarps) {
        const int blk = row_ids[bi];
        uint32_t kw[TPL][W], vw[TPL][W];
#pragma unroll
        for (int i = 0; i < TPL; ++i)
            load_chunk<D>(kv_row<D>(a.k_pool, blk, 2 * i + half, kh, Hkv), l16, kw[i]);
#pragma unroll
        for (int i = 0; i < TPL; ++i)
            load_chunk<D>(kv_row<D>(a.v_pool, blk, 2 * i + half, kh, Hkv), l16, vw[i]);

        // Partial logits: value index v = i * G + g (token 2i + half, head g).
        float acc[NV];
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
            float kf[DPL];
#pragma unroll
            for (int e = 0; e < W; ++e) {
                kf[2 * e] = bf_lo(kw[i][e]);
                kf[2 * e + 1] = bf_hi(kw[i][e]);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float t = 0.f;
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    t = fmaf(qv[g][d], kf[d], t);
                acc[i * G + g] = t;
            }
        }
        // Transposing butterfly over the 16 lanes of this half: each level keeps
        // the half of the values selected by the lane bit and adds the partner's.
        int n = NV;
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            const bool upper = (l16 & off) != 0;
            if (n > 1) {
                const int hn = n / 2;
#pragma unroll
                for (int j = 0; j < NV / 2; ++j) {
                    if (j < hn) {
                        const float send = upper ? acc[j] : acc[j + hn];
                        const float keep = upper ? acc[j + hn] : acc[j];
                        acc[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                n = hn;
            } else {
                acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
            }
        }
        // Now this lane holds KPL complete logits: token 2*(l16>>1) + half, heads
        // hbase .. hbase+KPL-1 with hbase = (l16 & 1) * KPL (G >= 2), or head 0 (G = 1).
        const int hbase = G >= 2 ? (l16 & 1) * KPL : 0;
        float bm[KPL];
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            float x = acc[k];
#pragma unroll
            for (int off = 2; off <= 16; off <<= 1)
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
            bm[k] = x;
        }
        // Every lane learns the block max of all G heads.
        float mx[G];
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            if (G >= 2) {
                const float other = __shfl_xor_sync(0xffffffffu, bm[k], 1);
                mx[k] = (l16 & 1) ? other : bm[k];
                mx[KPL + k < G ? KPL + k : k] = (l16 & 1) ? bm[k] : other;
            } else {
                mx[0] = bm[0];
            }
        }
        float mnew[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            mnew[g] = fmaxf(m_run[g], mx[g]);
            if (mnew[g] > m_run[g]) {                         // uniform across the warp
                const float f = ex2_approx(m_run[g] - mnew[g]);   // 0 when m_run = -inf
                l_part[g] *= f;
#pragma unroll
                for (int d = 0; d < DPL; ++d)
                    o[g][d] *= f;
                m_run[g] = mnew[g];
            }
        }
        float pk[KPL];
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            const int hg = hbase + k;
            pk[k] = ex2_approx(acc[k] - m_run[hg]);
            // in G = 1 the lane pair (l16, l16^1) holds the same value: count it once
            if (G >= 2 || (l16 & 1) == 0)
                l_part[hg] += pk[k];
        }
        // PV: lane owns columns [l16*DPL, +DPL) of its tokens 2i + half.
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
            float pv[G];
#pragma unroll
            for (int grp = 0; grp < (G >= 2 ? 2 : 1); ++grp) {
                const int src = half * 16 + 2 * i + grp;
#pragma unroll
                for (int k = 0; k < KPL; ++k)
                    pv[grp * KPL + k] = __shfl_sync(0xffffffffu, pk[k], src);
            }
#pragma unroll
            for (int e = 0; e < W; ++e) {
                const float v0 = bf_lo(vw[i][e]), v1 = bf_hi(vw[i][e]);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    o[g][2 * e] = fmaf(pv[g], v0, o[g][2 * e]);
                    o[g][2 * e + 1] = fmaf(pv[g], v1, o[g][2 * e + 1]);
                }
            }
        }
    }

    // Warp totals: l over all lanes, o over the two token halves.
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float x = l_part[g];
#pragma unroll
        for (int off = 1; off <= 16; off <<= 1)
            x += __shfl_xor_sync(0xffffffffu, x, off);
        l_part[g] = x;
#pragma unroll
        for (int d = 0; d < DPL; ++d)
            o[g][d] += __shfl_xor_sync(0xffffffffu, o[g][d], 16);
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            s_m[warp][g] = m_run[g];
            s_l[warp][g] = l_part[g];
        }
    }
    if (half == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < DPL; ++d)
                s_o[warp][g][l16 * DPL + d] = o[g][d];
    }
    __syncthreads();

    // Merge the warps with the incoming state (stored m is in natural-log units).
    __shared__ float s_min[G], s_lin[G];
    if (threadIdx.x < G) {
        const long long sh = static_cast<long long>(s) * Hq + kh * G + threadIdx.x;
        s_min[threadIdx.x] = a.m[sh] * kLog2e;
        s_lin[threadIdx.x] = a.l[sh];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
        const int g = e / D, d = e % D;
        const long long sh = static_cast<long long>(s) * Hq + kh * G + g;
        const float m_in = s_min[g];
        float mt = m_in;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mt = fmaxf(mt, s_m[w][g]);
        const float f_in = ex2_approx(m_in - mt);      // 0 for a fresh state (m_in = -inf)
        float acc_o = a.o[sh * D + d] * f_in;
        float acc_l = s_lin[g] * f_in;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = ex2_approx(s_m[w][g] - mt);
            acc_o = fmaf(s_o[w][g][d], f, acc_o);
            acc_l = fmaf(s_l[w][g], f, acc_l);
        }
        a.o[sh * D + d] = acc_o;
        if (d == 0) {
            a.l[sh] = acc_l;
            a.m[sh] = mt * kLn2;
        }
    }
}

__global__ void decode_init_kernel(float *m, float *l, float *o, long long n_state, int head_dim,
                                   int32_t *status)
{
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

template <int D, int G>
cudaError_t step_dg(const DecodeStepArgs &a, cudaStream_t stream)
{
    dim3 grid(a.num_kv_heads, a.num_seqs);
    decode_step_kernel<D, G><<<grid, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t step_d(const DecodeStepArgs &a, cudaStream_t stream)
{
    switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return step_dg<D, 1>(a, stream);
    case 2: return step_dg<D, 2>(a, stream);
    case 4: return step_dg<D, 4>(a, stream);
    case 8: return step_dg<D, 8>(a, stream);
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

cudaError_t launch_decode_init(float *m, float *l, float *o, int num_seqs, int num_q_heads,
                               int head_dim, int32_t *status, cudaStream_t stream)
{
    const long long n_state = static_cast<long long>(num_seqs) * num_q_heads;
    decode_init_kernel<<<grid_for(n_state * head_dim, 256), 256, 0, stream>>>(m, l, o, n_state,
                                                                             head_dim, status);
    return cudaGetLastError();
}

cudaError_t launch_decode_step(const DecodeStepArgs &a, cudaStream_t stream)
{
    switch (a.head_dim) {
    case 64: return step_d<64>(a, stream);
    case 128: return step_d<128>(a, stream);
    case 256: return step_d<256>(a, stream);
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
