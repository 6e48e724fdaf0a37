// noalloc.cu -- vfa_varlen_fwd_noalloc: the varlen forward with its scratch
// memory in a fixed array inside the library, for callers that cannot
// allocate device memory at all.
//
// Who needs it: code that runs where cudaMalloc is unavailable or not
// allowed -- a host callback or a real-time thread that must not block on
// the allocator, an inference runtime that hands kernels a fixed, pre-planned
// memory arena and forbids any other allocation, or a plugin that only ever
// sees the input and output pointers of its host framework.  Such callers
// cannot provide the workspace vfa_varlen_fwd asks for; this entry point
// supplies it from a static device array instead and otherwise runs the same
// scheduler and prefill kernels.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace {

// 1 MiB of scratch, reserved on every GPU that loads the library until the
// process exits.  It holds the forward's status word, work-list header and
// work list (32 bytes per item) plus the scheduler's per-sequence
// records; vfa_varlen_fwd_workspace_bytes() gives the size a problem needs.
constexpr size_t kStaticScratchBytes = 1u << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on `dev` (the current device), looked
// up once per device.  In host code the array's name only stands for the
// symbol; the kernels must be given this address.
void *scratch_address(int dev, cudaError_t *err)
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (*err != cudaSuccess)
            return nullptr;
        addr[dev] = p;
    }
    *err = cudaSuccess;
    return addr[dev];
}

}  // namespace

extern "C" vfa_status vfa_varlen_fwd_noalloc(const void *q, const void *k, const void *v,
                                             const int32_t *cu_seqlens_q,
                                             const int32_t *cu_seqlens_k, int total_q,
                                             int total_k, int max_seqlen_q, int batch,
                                             int num_heads, int num_kv_heads, int head_dim,
                                             float softmax_scale, int causal, int window_left,
                                             void *out, float *lse, int32_t *device_status,
                                             vfa_stream_t stream)
{
    char msg[256];
    const size_t need = vfa_varlen_fwd_workspace_bytes(batch, total_q, total_k, num_heads,
                                                       head_dim);
    if (need > kStaticScratchBytes) {
        snprintf(msg, sizeof msg,
                 "problem needs %zu bytes of scratch; the static scratch holds %zu "
                 "(use vfa_varlen_fwd with a caller workspace)",
                 need, kStaticScratchBytes);
        return vfa::set_error(VFA_ERR_UNSUPPORTED, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64)
        return vfa::set_error(VFA_ERR_CUDA, "cudaGetDevice failed");
    void *ws = scratch_address(dev, &e);
    if (ws == nullptr) {
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return vfa::set_error(VFA_ERR_CUDA, msg);
    }
    // The scheduler kernel rewrites the status word, the item count and the
    // fetch counter on every call, so nothing the previous call left behind
    // is read as input.
    vfa_status st = vfa_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, total_q, total_k,
                                   max_seqlen_q, batch, num_heads, num_kv_heads, head_dim,
                                   softmax_scale, causal, window_left, out, lse, ws,
                                   kStaticScratchBytes,
                                   stream);
    if (st != VFA_OK || device_status == nullptr)
        return st;
    e = cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "status copy failed: %s", cudaGetErrorString(e));
        return vfa::set_error(VFA_ERR_CUDA, msg);
    }
    return VFA_OK;
}
