// moe_static.cu -- moe_forward_static: the layer forward for callers that
// cannot allocate device memory.  Its scratch is one file-scope device array
// owned by the library; the caller passes only inputs and outputs.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "moe_layout.h"

namespace moe {
moe_status set_error(moe_status s, const char *msg);
moe_status check_forward_args(const moe_config *cfg, const moe_weights *w, const uint16_t *x,
                              const uint16_t *out, int rows);
}

namespace {

constexpr size_t kStaticWsBytes = MOE_STATIC_WORKSPACE_BYTES;

// Zero-initialised when the module loads; every GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void *g_static_addr[64];   // device address of g_static_ws, per device ordinal

// Device address of the array on the current device, looked up once per
// device (with that device current).  In host code `g_static_ws` names a
// host-side stand-in, never a device address.
moe_status static_ws_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return moe::set_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return moe::set_error(MOE_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p)
            return moe::set_error(MOE_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                                 : "null symbol address");
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_forward_static(const moe_config *cfg, const moe_weights *w,
                                         const uint16_t *x, uint16_t *out, int rows,
                                         void *stream) {
    // every argument check first: a refused call enqueues nothing
    moe_status s = moe::check_forward_args(cfg, w, x, out, rows);
    if (s != MOE_OK) return s;
    const moe::WsLayout L = moe::WsLayout::make(*cfg);
    if (L.total > kStaticWsBytes) {
        char msg[160];
        snprintf(msg, sizeof msg,
                 "configuration needs %zu workspace bytes; the static workspace holds %zu",
                 L.total, kStaticWsBytes);
        return moe::set_error(MOE_ERR_WORKSPACE, msg);
    }
    void *ws = nullptr;
    if ((s = static_ws_address(&ws)) != MOE_OK) return s;
    // The status word and the grid-barrier counter (the workspace header)
    // must start at zero; the rest of the scratch is written before it is
    // read.
    cudaError_t e = cudaMemsetAsync(ws, 0, L.ids, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return moe::set_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    return moe_forward(cfg, w, x, out, rows, ws, kStaticWsBytes, stream);
}
