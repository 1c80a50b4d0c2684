// noalloc.cu -- smoe_moe_forward_noalloc: the MoE layer forward with its
// workspace in a fixed device array that is part of the library image, for
// callers that have no way to allocate device memory (declared in
// include/smoe.h, which says who they are).
//
// The array is a file-scope __device__ variable: the CUDA driver reserves it
// on each device when the library's module is loaded there, so nothing in
// this file ever calls an allocator.  Each call clears the workspace's
// counter prefix with cudaMemsetAsync (a kernel-side store, no allocation)
// and then enqueues exactly what smoe_moe_forward enqueues.
#include <mutex>

#include "smoe.h"
#include "internal.h"

namespace {

static_assert(SMOE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// One workspace per device, shared by every call on that device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SMOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
void *g_scratch_ctx[kMaxDevices] = {nullptr};

// The driver's current context (cuCtxGetCurrent through the runtime's
// driver entry point, so the library needs no link to libcuda), or null.
void *current_context()
{
    using get_ctx_fn = int (*)(void **);
    static get_ctx_fn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<get_ctx_fn>(p);
    }();
    void *ctx = nullptr;
    if (!fn || fn(&ctx) != 0)
        return nullptr;
    return ctx;
}

// Device address of g_noalloc_scratch on the current device, looked up with
// that device current and cached per device together with the context it
// was looked up in: a new context (after a device reset) may have loaded the
// module, and with it the array, at another address.
smoe_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SMOE_ERR_CUDA;
    // null before the runtime has made the device's context current: the
    // lookup below then runs (and creates it), and the next call caches
    void *ctx = current_context();
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return SMOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return SMOE_OK;
}

}  // namespace

extern "C" smoe_status smoe_moe_forward_noalloc(const smoe_layer_desc *layer, const void *x,
                                                smoe_dtype x_dtype, int64_t num_tokens, float *y,
                                                int32_t *ids_out, float *w_out, void *cuda_stream)
{
    // 0 for an invalid layer description or a negative token count
    const size_t need = smoe_moe_workspace_bytes(layer, num_tokens);
    if (need == 0)
        return SMOE_ERR_INVALID_ARG;
    if (num_tokens == 0)  // nothing to enqueue; the forward checks the rest
        return smoe_moe_forward(layer, x, x_dtype, 0, y, nullptr, 0, ids_out, w_out,
                                cuda_stream);
    // the forward's own pointer and device checks, repeated so that a call
    // that fails them enqueues nothing (not even the memset below)
    if ((x_dtype != SMOE_F32 && x_dtype != SMOE_BF16) || !x || !y ||
        reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16)
        return SMOE_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SMOE_ERR_CUDA;
    if (major != 10 || minor != 3)
        return SMOE_ERR_UNSUPPORTED;
    if (need > static_cast<size_t>(SMOE_NOALLOC_SCRATCH_BYTES))
        return SMOE_ERR_WORKSPACE;
    void *scratch = nullptr;
    const smoe_status st = scratch_address(&scratch);
    if (st != SMOE_OK)
        return st;
    // A previous call may have used the same bytes for another layer shape
    // (different counter offsets) or may have stopped on an error, so the
    // counters are cleared on every call rather than once.
    const size_t zero = smoe::moe_workspace_zero_bytes(layer, num_tokens);
    if (cudaMemsetAsync(scratch, 0, zero, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return SMOE_ERR_CUDA;
    return smoe_moe_forward(layer, x, x_dtype, num_tokens, y, scratch, need, ids_out, w_out,
                            cuda_stream);
}
