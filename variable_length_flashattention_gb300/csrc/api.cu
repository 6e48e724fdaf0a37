// api.cu -- the C ABI declared in include/vfa.h: argument checks, TMA tensor
// map encoding, workspace carve-up and launches.  Nothing here allocates or
// frees device memory.
#include <algorithm>
#include <cfloat>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

thread_local char g_err[512] = "";

vfa_status fail(vfa_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

vfa_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(VFA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceInfo {
    bool ok = false;
    int sm_count = 0;
    int major = 0, minor = 0;
};

// The current device must be compute capability 10.3 (the only one built for).
vfa_status current_device(DeviceInfo *out)
{
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(VFA_ERR_CUDA, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!cache[dev].ok) {
            DeviceInfo d;
            if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) ||
                (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
                (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)))
                return cuda_fail(e, "cudaDeviceGetAttribute");
            d.ok = true;
            cache[dev] = d;
        }
        *out = cache[dev];
    }
    if (out->major != 10 || out->minor != 3)
        return fail(VFA_ERR_ARCH, "device is sm_%d%d; this library is built for sm_103a only",
                    out->major, out->minor);
    return VFA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

vfa_status get_encoder(EncodeTiledFn *fn)
{
    static std::once_flag once;
    static EncodeTiledFn f = nullptr;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                               cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            f = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!f)
        return fail(VFA_ERR_CUDA, "cuTensorMapEncodeTiled is not available (%s)",
                    cudaGetErrorName(err));
    *fn = f;
    return VFA_OK;
}

// [rows, heads, head_dim] tensor of bf16 (elem_bytes 2) or 8-bit codes
// (elem_bytes 1) as a 3-D TMA map (innermost first: dim, head, row); box =
// 128 bytes of columns x 1 head x box_rows rows, 128-byte swizzle -- or, for
// rows of only 64 bytes (8-bit codes at head_dim 64), 64 bytes with the
// 64-byte swizzle.
vfa_status encode_packed_map(CUtensorMap *map, const void *base, int rows, int heads,
                             int head_dim, int box_rows, int elem_bytes = 2)
{
    EncodeTiledFn enc;
    vfa_status st = get_encoder(&enc);
    if (st)
        return st;
    const cuuint64_t eb = static_cast<cuuint64_t>(elem_bytes);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * eb,
                                   static_cast<cuuint64_t>(heads) * head_dim * eb};
    const int box_bytes = head_dim * elem_bytes >= 128 ? 128 : 64;
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_bytes / elem_bytes), 1,
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map,
                     elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(VFA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return VFA_OK;
}

// The bf16 output [rows, heads, head_dim] as a 3-D TMA map for tile stores:
// boxes of 32 columns (64 bytes) x 1 head x 32 rows, 64-byte swizzle -- one
// prefill warp's 32 rows of a 32-column chunk, as it stages them.
vfa_status encode_out_map(CUtensorMap *map, void *base, int rows, int heads, int head_dim)
{
    EncodeTiledFn enc;
    vfa_status st = get_encoder(&enc);
    if (st)
        return st;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                   static_cast<cuuint64_t>(heads) * head_dim * 2};
    const cuuint32_t box[3] = {32, 1, 32};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(VFA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return VFA_OK;
}

// [num_blocks * block_size tokens, kv_heads, head_dim] bf16 pool as the same
// kind of 3-D TMA map as the packed tensors: one box is 64 columns of one
// block's block_size token rows for one kv head.
vfa_status encode_pool_map(CUtensorMap *map, const void *base, int num_blocks, int block_size,
                           int kv_heads, int head_dim)
{
    return encode_packed_map(map, base, num_blocks * block_size, kv_heads, head_dim, block_size);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

// Most runs a split decode step cuts a tile into (the merge keeps one weight
// per run and q head in the step kernel's 48 KB of shared memory).
constexpr int kMaxDecodeSplits = 1024;

}  // namespace

vfa_status vfa::set_error(vfa_status st, const char *message)
{
    return fail(st, "%s", message);
}

extern "C" {

const char *vfa_last_error(void) { return g_err; }

const char *vfa_version(void) { return "vfa 0.1 sm_103a"; }

size_t vfa_varlen_fwd_workspace_bytes(int batch, int total_q, int total_k, int num_heads,
                                      int head_dim)
{
    if (batch < 1 || total_q < 0 || total_k < 0 || num_heads < 1 || !supported_head_dim(head_dim))
        return 0;
    return vfa::workspace_layout(batch, total_q, total_k, num_heads, vfa::kBlockQ,
                                 vfa::block_k_for(head_dim))
        .total_bytes;
}

vfa_status vfa_varlen_fwd_tile_shape(int head_dim, int *block_q, int *block_k, int *pair_tiles)
{
    if (!supported_head_dim(head_dim))
        return fail(VFA_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", head_dim);
    if (!block_q || !block_k || !pair_tiles)
        return fail(VFA_ERR_INVALID_ARG, "null output pointer");
    *block_q = vfa::kBlockQ;
    *block_k = vfa::block_k_for(head_dim);
    *pair_tiles = vfa::pairs_for(head_dim) ? 1 : 0;
    return VFA_OK;
}

vfa_status vfa_varlen_schedule(const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                               int total_q, int total_k, int max_seqlen_q, int batch,
                               int num_heads, int block_q, int block_k, int causal,
                               int window_left, int pair_tiles, int32_t *items,
                               int items_capacity,
                               int32_t *n_items, int32_t *status, void *scratch,
                               size_t scratch_bytes, vfa_stream_t stream)
{
    if (!cu_seqlens_q || !cu_seqlens_k || !items || !n_items || !status || !scratch)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (batch < 1 || num_heads < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
        block_q < 1 || block_k < 1 || items_capacity < 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument");
    if (causal < 0 || causal > 2)
        return fail(VFA_ERR_INVALID_ARG, "causal must be 0, 1 (top-left) or 2 (bottom-right)");
    if (window_left >= 0 && causal == 0)
        return fail(VFA_ERR_INVALID_ARG, "a sliding window needs a causal mode");
    if (!aligned(items, 16) || !aligned(scratch, 8))
        return fail(VFA_ERR_INVALID_ARG, "items must be 16-byte and scratch 8-byte aligned");
    if ((block_k & (block_k - 1)) != 0 || block_q % block_k != 0)
        return fail(VFA_ERR_UNSUPPORTED,
                    "block_k must be a power of two and block_q a multiple of it (%d, %d)",
                    block_q, block_k);
    const int need = vfa::schedule_scratch_ints(batch, total_q, total_k, block_q, block_k);
    if (scratch_bytes < static_cast<size_t>(need) * sizeof(int))
        return fail(VFA_ERR_INVALID_ARG, "scratch too small: %zu < %zu bytes", scratch_bytes,
                    static_cast<size_t>(need) * sizeof(int));
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    vfa::SchedArgs a;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.batch = batch;
    a.total_q = total_q;
    a.total_k = total_k;
    a.max_seqlen_q = max_seqlen_q;
    a.num_heads = num_heads;
    a.block_q = block_q;
    a.block_k = block_k;
    a.causal = causal;
    a.window_left = window_left < 0 ? -1 : window_left;
    a.pair = pair_tiles != 0;
    a.items = reinterpret_cast<int4 *>(items);
    a.item_capacity = items_capacity;
    a.n_items = n_items;
    a.status = status;
    a.next_item = nullptr;
    a.scratch = static_cast<int32_t *>(scratch);
    a.scratch_ints = static_cast<int>(scratch_bytes / sizeof(int));
    cudaError_t e = vfa::launch_schedule(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "scheduler launch");
    return VFA_OK;
}

// The forward for bf16 q, k (qk_fp8 = 0) or FP8 E4M3 q, k codes with
// per-tensor descales (qk_fp8 = 1, head_dim 128).
static vfa_status varlen_fwd_impl(const void *q, const void *k, const void *v,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  int total_q, int total_k, int max_seqlen_q, int batch,
                                  int num_heads, int num_kv_heads, int head_dim,
                                  float softmax_scale, int causal, int window_left, void *out,
                                  float *lse, void *workspace, size_t workspace_bytes,
                                  vfa_stream_t stream, int qk_fp8, float descale_q,
                                  float descale_k)
{
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out || !lse || !workspace)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (batch < 1 || num_heads < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument (batch %d, heads %d, totals %d/%d)",
                    batch, num_heads, total_q, total_k);
    if (num_kv_heads < 1 || num_heads % num_kv_heads != 0)
        return fail(VFA_ERR_INVALID_ARG, "num_heads %d is not a multiple of num_kv_heads %d",
                    num_heads, num_kv_heads);
    if (causal < 0 || causal > 2)
        return fail(VFA_ERR_INVALID_ARG, "causal must be 0, 1 (top-left) or 2 (bottom-right)");
    if (window_left >= 0 && causal == 0)
        return fail(VFA_ERR_INVALID_ARG, "a sliding window needs a causal mode");
    if (!supported_head_dim(head_dim))
        return fail(VFA_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", head_dim);
    if (!(softmax_scale >= 0.f) || softmax_scale > FLT_MAX)
        return fail(VFA_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0 (got %g)",
                    static_cast<double>(softmax_scale));
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 256))
        return fail(VFA_ERR_INVALID_ARG,
                    "q, k, v, out must be 16-byte aligned, lse 4-byte, workspace 256-byte");
    if (static_cast<long long>(num_heads) * head_dim * 2 > (1LL << 40) ||
        static_cast<long long>(total_q) * num_heads > (1LL << 31) ||
        static_cast<long long>(total_k) * num_heads > (1LL << 31))
        return fail(VFA_ERR_UNSUPPORTED, "tensor too large");
    const int bq = vfa::kBlockQ, bk = vfa::block_k_for(head_dim);
    const vfa::WorkspaceLayout wl =
        vfa::workspace_layout(batch, total_q, total_k, num_heads, bq, bk);
    if (workspace_bytes < wl.total_bytes)
        return fail(VFA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    wl.total_bytes);
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    int32_t *n_items = reinterpret_cast<int32_t *>(ws + 4);
    int32_t *next_item = reinterpret_cast<int32_t *>(ws + 8);
    int4 *items = reinterpret_cast<int4 *>(ws + wl.items_offset);

    vfa::SchedArgs sa;
    sa.cu_q = cu_seqlens_q;
    sa.cu_k = cu_seqlens_k;
    sa.batch = batch;
    sa.total_q = total_q;
    sa.total_k = total_k;
    sa.max_seqlen_q = max_seqlen_q;
    sa.num_heads = num_heads;
    sa.block_q = bq;
    sa.block_k = bk;
    sa.causal = causal;
    sa.window_left = window_left < 0 ? -1 : window_left;
    sa.pair = vfa::pairs_for(head_dim) ? 1 : 0;
    sa.items = items;
    sa.item_capacity = wl.item_capacity;
    sa.n_items = n_items;
    sa.status = status;
    sa.next_item = next_item;
    sa.scratch = reinterpret_cast<int32_t *>(ws + wl.scratch_offset);
    sa.scratch_ints = wl.scratch_ints;
    cudaError_t e = vfa::launch_schedule(sa, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "scheduler launch");

    if (wl.item_capacity == 0)
        return VFA_OK;                       // no query rows at all

    vfa::PrefillArgs pa;
    memset(&pa, 0, sizeof pa);
    const int qk_bytes = qk_fp8 ? 1 : 2;
    if ((st = encode_packed_map(&pa.tm_q, q, total_q, num_heads, head_dim, bq, qk_bytes)) ||
        (st = encode_packed_map(&pa.tm_k, k, total_k, num_kv_heads, head_dim, bk, qk_bytes)) ||
        (st = encode_packed_map(&pa.tm_v, v, total_k, num_kv_heads, head_dim, bk)) ||
        (st = encode_out_map(&pa.tm_o, out, total_q, num_heads, head_dim)))
        return st;
    pa.cu_q = cu_seqlens_q;
    pa.cu_k = cu_seqlens_k;
    pa.items = items;
    pa.n_items = n_items;
    pa.next_item = next_item;
    pa.status = status;
    pa.out = out;
    pa.lse = lse;
    pa.num_heads = num_heads;
    pa.kv_group = num_heads / num_kv_heads;
    // The kernel takes row maxima on raw scores, which needs a positive scale;
    // a zero scale (uniform weights) becomes the smallest normal float, which
    // gives the same weights for every finite score.
    pa.scale_log2 = softmax_scale > 0.f ? softmax_scale * 1.4426950408889634f : FLT_MIN;
    if (qk_fp8) {
        // S = descale_q * descale_k * (codes of q) . (codes of k)
        const double sl = static_cast<double>(softmax_scale) * descale_q * descale_k *
                          1.4426950408889634;
        pa.scale_log2 = sl > 0.0 ? static_cast<float>(sl) : FLT_MIN;
    }
    pa.qk_fp8 = qk_fp8;
    pa.causal = causal;
    pa.window_left = sa.window_left;
    const int grid = wl.item_capacity < dev.sm_count ? wl.item_capacity : dev.sm_count;
    e = vfa::launch_prefill(head_dim, pa, grid, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "prefill launch");
    return VFA_OK;
}

vfa_status vfa_varlen_fwd(const void *q, const void *k, const void *v,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int total_q,
                          int total_k, int max_seqlen_q, int batch, int num_heads,
                          int num_kv_heads, int head_dim, float softmax_scale, int causal,
                          int window_left, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, vfa_stream_t stream)
{
    return varlen_fwd_impl(q, k, v, cu_seqlens_q, cu_seqlens_k, total_q, total_k, max_seqlen_q,
                           batch, num_heads, num_kv_heads, head_dim, softmax_scale, causal,
                           window_left, out, lse, workspace, workspace_bytes, stream, 0, 1.f, 1.f);
}

vfa_status vfa_varlen_fwd_fp8(const void *q_fp8, const void *k_fp8, const void *v,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                              int total_q, int total_k, int max_seqlen_q, int batch,
                              int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                              float descale_q, float descale_k, int causal, int window_left,
                              void *out, float *lse, void *workspace, size_t workspace_bytes,
                              vfa_stream_t stream)
{
    if (!supported_head_dim(head_dim))
        return fail(VFA_ERR_UNSUPPORTED, "FP8 forward head_dim %d not supported (64, 128, 256)",
                    head_dim);
    if (!(descale_q > 0.f) || !(descale_k > 0.f) || descale_q > FLT_MAX || descale_k > FLT_MAX)
        return fail(VFA_ERR_INVALID_ARG, "descale_q and descale_k must be finite and > 0");
    return varlen_fwd_impl(q_fp8, k_fp8, v, cu_seqlens_q, cu_seqlens_k, total_q, total_k,
                           max_seqlen_q, batch, num_heads, num_kv_heads, head_dim, softmax_scale,
                           causal, window_left, out, lse, workspace, workspace_bytes, stream, 1,
                           descale_q, descale_k);
}

size_t vfa_varlen_bwd_workspace_bytes(int batch, int total_q, int num_heads, int head_dim)
{
    if (batch < 1 || total_q < 0 || num_heads < 1 || !supported_head_dim(head_dim))
        return 0;
    return vfa::bwd_workspace_bytes(batch, total_q, num_heads, head_dim);
}

vfa_status vfa_varlen_bwd(const void *q, const void *k, const void *v, const void *out,
                          const void *dout, const float *lse, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, int total_q, int total_k, int batch,
                          int num_heads, int num_kv_heads, int head_dim, float softmax_scale,
                          int causal, int window_left, void *dq, void *dk, void *dv,
                          void *workspace, size_t workspace_bytes, vfa_stream_t stream)
{
    if (!q || !k || !v || !out || !dout || !lse || !cu_seqlens_q || !cu_seqlens_k || !dq ||
        !dk || !dv || !workspace)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (batch < 1 || num_heads < 1 || total_q < 0 || total_k < 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument (batch %d, heads %d, totals %d/%d)",
                    batch, num_heads, total_q, total_k);
    if (num_kv_heads < 1 || num_heads % num_kv_heads != 0)
        return fail(VFA_ERR_INVALID_ARG, "num_heads %d is not a multiple of num_kv_heads %d",
                    num_heads, num_kv_heads);
    if (causal < 0 || causal > 2)
        return fail(VFA_ERR_INVALID_ARG, "causal must be 0, 1 (top-left) or 2 (bottom-right)");
    if (window_left >= 0 && causal == 0)
        return fail(VFA_ERR_INVALID_ARG, "a sliding window needs a causal mode");
    if (!supported_head_dim(head_dim))
        return fail(VFA_ERR_UNSUPPORTED, "backward head_dim %d not supported (64, 128, 256)",
                    head_dim);
    if (!(softmax_scale > 0.f) || softmax_scale > FLT_MAX)
        return fail(VFA_ERR_INVALID_ARG, "softmax_scale must be finite and > 0 (got %g)",
                    static_cast<double>(softmax_scale));
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 256))
        return fail(VFA_ERR_INVALID_ARG,
                    "tensors must be 16-byte aligned, lse 4-byte, workspace 256-byte");
    if (static_cast<long long>(total_q) * num_heads * head_dim > (1LL << 31) ||
        static_cast<long long>(total_k) * num_heads > (1LL << 31))
        return fail(VFA_ERR_UNSUPPORTED, "tensor too large");
    const size_t need = vfa::bwd_workspace_bytes(batch, total_q, num_heads, head_dim);
    if (workspace_bytes < need)
        return fail(VFA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    need);
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    vfa::BwdArgs a;
    memset(&a, 0, sizeof a);
    const int box = vfa::bwd_step_rows(head_dim), box_kv = vfa::bwd_dq_step_rows(head_dim);
    const int box_q = vfa::bwd_kv_step_rows(head_dim);
    if ((st = encode_packed_map(&a.tm_q, q, total_q, num_heads, head_dim, box)) ||
        (st = encode_packed_map(&a.tm_do, dout, total_q, num_heads, head_dim, box)) ||
        (st = encode_packed_map(&a.tm_k, k, total_k, num_kv_heads, head_dim, box)) ||
        (st = encode_packed_map(&a.tm_v, v, total_k, num_kv_heads, head_dim, box)) ||
        (st = encode_packed_map(&a.tm_ks, k, total_k, num_kv_heads, head_dim, box_kv)) ||
        (st = encode_packed_map(&a.tm_vs, v, total_k, num_kv_heads, head_dim, box_kv)) ||
        (st = encode_packed_map(&a.tm_qs, q, total_q, num_heads, head_dim, box_q)) ||
        (st = encode_packed_map(&a.tm_dos, dout, total_q, num_heads, head_dim, box_q)))
        return st;
    vfa::bwd_workspace_split(workspace, batch, total_q, num_heads, &a);
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.batch = batch;
    a.total_q = total_q;
    a.total_k = total_k;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.scale = softmax_scale;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.causal = causal;
    a.window_left = window_left < 0 ? -1 : window_left;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int key_tile_bound = total_k / 128 + batch;
    const int q_tile_bound = total_q / 128 + batch;
    cudaError_t e = vfa::launch_bwd(head_dim, a, key_tile_bound, q_tile_bound, dev.sm_count, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward launch");
    return VFA_OK;
}

vfa_status vfa_paged_decode_init(float *m, float *l, float *o, int num_seqs, int num_q_heads,
                                 int head_dim, int32_t *device_status, vfa_stream_t stream)
{
    if (!m || !l || !o)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (num_seqs < 1 || num_q_heads < 1 || head_dim < 1)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument");
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    cudaError_t e = vfa::launch_decode_init(m, l, o, num_seqs, num_q_heads, head_dim,
                                            device_status, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "decode init launch");
    return VFA_OK;
}

static vfa_status check_decode_args(const void *q, const void *k_pool, const void *v_pool,
                                    int num_blocks, const int32_t *tile_blocks,
                                    const int32_t *counts, int tile_capacity, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size)
{
    if (!k_pool || !v_pool || !tile_blocks || !counts || (q == nullptr && num_q_heads < 0))
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_blocks < 0 ||
        tile_capacity < 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument");
    if (num_q_heads % num_kv_heads != 0)
        return fail(VFA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, num_kv_heads);
    const int g = num_q_heads / num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(VFA_ERR_UNSUPPORTED, "q heads per kv head %d not supported (1, 2, 4, 8)", g);
    if (!supported_head_dim(head_dim))
        return fail(VFA_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", head_dim);
    if (block_size != 16)
        return fail(VFA_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
    if (num_blocks > (1 << 26))
        return fail(VFA_ERR_UNSUPPORTED, "num_blocks %d above 2^26 not supported", num_blocks);
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || (q && !aligned(q, 16)) ||
        !aligned(tile_blocks, 4) || !aligned(counts, 4))
        return fail(VFA_ERR_INVALID_ARG, "pools and q must be 16-byte aligned");
    return VFA_OK;
}

static vfa_status decode_step_impl(const void *q, const void *k_pool, const void *v_pool,
                                   int num_blocks, const int32_t *tile_blocks,
                                   const int32_t *tile_block_counts,
                                   const int32_t *tile_token_counts, int tile_capacity,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float softmax_scale, float *m, float *l,
                                   float *o, int32_t *device_status, int num_splits,
                                   void *workspace, size_t workspace_bytes, vfa_stream_t stream)
{
    if (!q || !m || !l || !o)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (!std::isfinite(softmax_scale))
        return fail(VFA_ERR_INVALID_ARG, "softmax_scale must be finite");
    if (tile_token_counts && !aligned(tile_token_counts, 4))
        return fail(VFA_ERR_INVALID_ARG, "tile_token_counts must be 4-byte aligned");
    vfa_status st = check_decode_args(q, k_pool, v_pool, num_blocks, tile_blocks,
                                      tile_block_counts, tile_capacity, num_seqs, num_q_heads,
                                      num_kv_heads, head_dim, block_size);
    if (st)
        return st;
    if (!aligned(o, 16) || !aligned(m, 4) || !aligned(l, 4))
        return fail(VFA_ERR_INVALID_ARG, "o must be 16-byte aligned");
    DeviceInfo dev;
    if ((st = current_device(&dev)))
        return st;
    vfa::DecodeStepArgs a;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.tile_blocks = tile_blocks;
    a.tile_block_counts = tile_block_counts;
    a.num_blocks = num_blocks;
    a.tile_capacity = tile_capacity;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.m = m;
    a.l = l;
    a.o = o;
    a.status = device_status;
    a.tile_token_counts = tile_token_counts;
    a.num_splits = 1;
    a.part = nullptr;
    a.tickets = nullptr;
    if (num_splits > 1) {
        a.num_splits = num_splits;
        vfa::decode_split_workspace_carve(workspace, num_seqs, num_kv_heads, &a);
    }
    a.scale_log2 = static_cast<float>(
        (softmax_scale > 0.f ? static_cast<double>(softmax_scale) : 1.0 / std::sqrt(double(head_dim))) *
        1.4426950408889634);
    vfa::DecodeMaps maps;
    if ((st = encode_pool_map(&maps.tm_k, k_pool, num_blocks, block_size, num_kv_heads,
                              head_dim)) ||
        (st = encode_pool_map(&maps.tm_v, v_pool, num_blocks, block_size, num_kv_heads,
                              head_dim)))
        return st;
    cudaError_t e = vfa::launch_decode_step(a, maps, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "decode step launch");
    return VFA_OK;
}

vfa_status vfa_paged_decode_step(const void *q, const void *k_pool, const void *v_pool,
                                 int num_blocks, const int32_t *tile_blocks,
                                 const int32_t *tile_block_counts,
                                 const int32_t *tile_token_counts, int tile_capacity,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, float softmax_scale, float *m, float *l,
                                 float *o, int32_t *device_status, vfa_stream_t stream)
{
    return decode_step_impl(q, k_pool, v_pool, num_blocks, tile_blocks, tile_block_counts,
                            tile_token_counts, tile_capacity, num_seqs, num_q_heads,
                            num_kv_heads, head_dim, block_size, softmax_scale, m, l, o,
                            device_status, 1, nullptr, 0, stream);
}

size_t vfa_paged_decode_split_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, int num_splits)
{
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads ||
        !supported_head_dim(head_dim) || num_splits < 1 || num_splits > kMaxDecodeSplits)
        return 0;
    return vfa::decode_split_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             num_splits);
}

vfa_status vfa_paged_decode_split_count(int num_seqs, int num_kv_heads, int tile_capacity,
                                        int *num_splits)
{
    if (!num_splits)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (num_seqs < 1 || num_kv_heads < 1 || tile_capacity < 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument");
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    // four step CTAs fit on an SM: aim for that many CTAs on every SM, with
    // runs of at least eight blocks
    const long long rows = static_cast<long long>(num_seqs) * num_kv_heads;
    long long n = (4LL * dev.sm_count + rows - 1) / rows;
    n = std::min<long long>(n, std::max(1, tile_capacity / 8));
    n = std::max<long long>(1, std::min<long long>(n, kMaxDecodeSplits));
    *num_splits = static_cast<int>(n);
    return VFA_OK;
}

vfa_status vfa_paged_decode_step_split(const void *q, const void *k_pool, const void *v_pool,
                                       int num_blocks, const int32_t *tile_blocks,
                                       const int32_t *tile_block_counts,
                                       const int32_t *tile_token_counts, int tile_capacity,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float softmax_scale,
                                       float *m, float *l, float *o, int32_t *device_status,
                                       int num_splits, void *workspace, size_t workspace_bytes,
                                       vfa_stream_t stream)
{
    if (num_splits < 1 || num_splits > kMaxDecodeSplits)
        return fail(VFA_ERR_INVALID_ARG, "num_splits %d outside [1, %d]", num_splits,
                    kMaxDecodeSplits);
    if (num_splits > 1) {
        if (!workspace || !aligned(workspace, 256))
            return fail(VFA_ERR_INVALID_ARG, "workspace must be a non-null, 256-byte aligned "
                                             "pointer");
        if (num_seqs < 1 || num_kv_heads < 1 || num_q_heads < 1)
            return fail(VFA_ERR_INVALID_ARG, "bad size argument");
        const size_t need = vfa_paged_decode_split_workspace_bytes(num_seqs, num_q_heads,
                                                                   num_kv_heads, head_dim,
                                                                   num_splits);
        if (need == 0)
            return fail(VFA_ERR_UNSUPPORTED, "no split workspace for these sizes");
        if (workspace_bytes < need)
            return fail(VFA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes",
                        workspace_bytes, need);
    }
    return decode_step_impl(q, k_pool, v_pool, num_blocks, tile_blocks, tile_block_counts,
                            tile_token_counts, tile_capacity, num_seqs, num_q_heads,
                            num_kv_heads, head_dim, block_size, softmax_scale, m, l, o,
                            device_status, num_splits, workspace, workspace_bytes, stream);
}

vfa_status vfa_paged_decode_finalize(const float *l, const float *o, int num_seqs,
                                     int num_q_heads, int head_dim, void *out,
                                     vfa_stream_t stream)
{
    if (!l || !o || !out)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    if (num_seqs < 1 || num_q_heads < 1 || head_dim < 8 || head_dim % 8 != 0)
        return fail(VFA_ERR_INVALID_ARG, "bad size argument (head_dim must be a multiple of 8)");
    if (!aligned(o, 16) || !aligned(out, 16))
        return fail(VFA_ERR_INVALID_ARG, "o and out must be 16-byte aligned");
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    cudaError_t e = vfa::launch_decode_finalize(l, o, num_seqs, num_q_heads, head_dim, out,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "decode finalize launch");
    return VFA_OK;
}

vfa_status vfa_debug_bounded_wait(int32_t *device_status, vfa_stream_t stream)
{
    if (!device_status || !aligned(device_status, 4))
        return fail(VFA_ERR_INVALID_ARG, "device_status must be a non-null, aligned pointer");
    DeviceInfo dev;
    vfa_status st = current_device(&dev);
    if (st)
        return st;
    cudaError_t e = vfa::launch_debug_bounded_wait(device_status,
                                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "bounded-wait hook launch");
    return VFA_OK;
}

vfa_status vfa_debug_paged_gather(const void *k_pool, const void *v_pool, int num_blocks,
                                  const int32_t *tile_blocks, const int32_t *tile_block_counts,
                                  int tile_capacity, int num_seqs, int num_kv_heads, int head_dim,
                                  int block_size, void *k_out, void *v_out,
                                  int32_t *device_status, vfa_stream_t stream)
{
    if (!k_out || !v_out)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    vfa_status st = check_decode_args(nullptr, k_pool, v_pool, num_blocks, tile_blocks,
                                      tile_block_counts, tile_capacity, num_seqs, num_kv_heads,
                                      num_kv_heads, head_dim, block_size);
    if (st)
        return st;
    if (!aligned(k_out, 16) || !aligned(v_out, 16))
        return fail(VFA_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    DeviceInfo dev;
    if ((st = current_device(&dev)))
        return st;
    vfa::DecodeStepArgs a;
    memset(&a, 0, sizeof a);
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.tile_blocks = tile_blocks;
    a.tile_block_counts = tile_block_counts;
    a.num_blocks = num_blocks;
    a.tile_capacity = tile_capacity;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_kv_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.status = device_status;
    cudaError_t e =
        vfa::launch_decode_gather(a, k_out, v_out, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "decode gather launch");
    return VFA_OK;
}

vfa_status vfa_read_status(const void *device_status_word, vfa_stream_t stream,
                           int32_t *host_status)
{
    if (!device_status_word || !host_status)
        return fail(VFA_ERR_INVALID_ARG, "null pointer argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(host_status, device_status_word, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy (status)");
    return VFA_OK;
}

}  // extern "C"
