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

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Identifier of the calling thread's current CUDA context (unique within the
// process: a context created after cudaDeviceReset gets a new one).  False
// when no context is current or the driver does not offer the query.
bool current_context_id(unsigned long long *id)
{
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_scratch on `dev` (the current device).  In host
// code the array's name only stands for the symbol; the kernels must be given
// this address.  It is looked up once per device and context: the cache
// remembers which context the address belongs to, and a call made under
// another context (after cudaDeviceReset, or from a thread with its own
// context) looks the address up again instead of reusing a dead one.
void *scratch_address(int dev, cudaError_t *err)
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] != nullptr && have_id && ctx_of[dev] == id) {
        *err = cudaSuccess;
        return addr[dev];
    }
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (*err != cudaSuccess)
        return nullptr;
    // the look-up makes the device's primary context current if none was
    unsigned long long id_now = 0;
    if (current_context_id(&id_now)) {
        addr[dev] = p;
        ctx_of[dev] = id_now;
    } else {
        addr[dev] = nullptr;      // no way to tell contexts apart: look up on every call
    }
    return p;
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
