// conv_stack_forward_noalloc: the layer-stack driver with its intermediate activations held in a
// buffer that is part of the library image instead of a workspace the caller allocates.
//
// Who needs it: code that may not allocate device memory at run time - a plug-in running inside a
// host framework that owns every allocation, a real-time or safety-certified pipeline that forbids
// allocation after start-up, or a caller whose memory is fully reserved by its own pool - yet
// still wants to run a multi-layer stack, whose layer-to-layer activations need scratch space.
//
// The scratch is one file-scope device array of X3_NOALLOC_SCRATCH_BYTES. Every GPU that loads the
// library holds it until the process exits, and every call on a device shares it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace x3 {

static __device__ __align__(256) unsigned char g_noalloc_scratch[X3_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kMaxDevices];
static void* g_noalloc_ctx[kMaxDevices];  // the context the address was resolved in

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The calling thread's current context (NULL if the driver entry point is unavailable).
static void* current_context() {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        fn = (CtxGetCurrentFn)f;
    }
    CUcontext c = nullptr;
    return fn(&c) == CUDA_SUCCESS ? (void*)c : nullptr;
}

// Device address of the scratch array on the current device. The array's name is only a host-side
// stand-in in host code, so its address is looked up with that device current: once per device and
// context (again after a cudaDeviceReset or under another context, whose module instance is a
// different allocation).
static x3_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(X3_ERR_CUDA, "conv_stack_forward_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(X3_ERR_UNSUPPORTED, "conv_stack_forward_noalloc: device %d out of range", dev);
    void* ctx = current_context();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || !ctx || g_noalloc_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(X3_ERR_CUDA, "conv_stack_forward_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = current_context();  // the runtime has made the device's context current by now
    }
    *out = g_noalloc_ptr[dev];
    return X3_OK;
}

}  // namespace x3

using namespace x3;

extern "C" x3_status conv_stack_forward_noalloc(const x3_conv_plan* const* plans, int n_layers, const void* x,
                                                void* const* carries, int carry_valid,
                                                const void* const* w_packed, const void* const* bias, void* y,
                                                x3_stream_t stream) {
    if (!plans || n_layers < 1) return fail(X3_ERR_INVALID, "conv_stack_forward_noalloc: no layers");
    const size_t need = conv_stack_workspace_bytes(plans, n_layers);
    if (need > (size_t)X3_NOALLOC_SCRATCH_BYTES)
        return fail(X3_ERR_OOM,
                    "conv_stack_forward_noalloc: these layers need %zu bytes of scratch for their intermediate "
                    "activations; the built-in scratch holds %zu bytes (use conv_stack_forward with a workspace)",
                    need, (size_t)X3_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    if (need) {
        x3_status st = noalloc_scratch(&scratch);
        if (st != X3_OK) return st;
    }
    // Every intermediate element is written by its layer before the next layer reads it, so nothing
    // left in the scratch by an earlier call has to be cleared.
    return conv_stack_forward(plans, n_layers, x, carries, carry_valid, w_packed, bias, y, scratch,
                              need ? (size_t)X3_NOALLOC_SCRATCH_BYTES : 0, stream);
}
