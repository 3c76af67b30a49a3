// gdn_noalloc.cu -- gdn_decode_conv_norm_noalloc: the fused decode from the
// projections (gdn_decode_conv_norm) for callers that cannot hand the library
// a workspace.
//
// Who cannot allocate, and why.  gdn_decode_conv_norm needs batch*NK int32
// counters of device memory beyond its inputs and outputs (the last CTA to
// read a key head's q/k conv-ring rows is the one that writes them back).  A
// caller that owns no device allocator (a plain C host that only receives
// tensor pointers from elsewhere), one whose memory plan is fixed before the
// decode loop starts and may not grow, or one that must not stall the device
// (cudaFree waits until the device is idle) has no good way to produce that
// buffer.  This entry point brings its own: a fixed,
// modest array of counters in the library's static device memory, so the
// call itself allocates nothing and frees nothing.
//
// How.  The counters live in `g_noalloc_counters` below (zero-initialised
// when the module is loaded on a device; every completed call leaves the ones
// it used at zero again, so they start at zero for the next call).  Its
// device address is looked up with cudaGetSymbolAddress once per device, the
// first time a call runs with that device current, and cached.  The call
// runs the argument checks of gdn_decode_conv_norm first (a rejected or empty
// call makes no CUDA call), then looks the address up and launches with it as
// the workspace, so the arithmetic and kernels are exactly those of the
// workspace entry point.
//
// Limits.  batch * NK <= GDN_NOALLOC_MAX_KEY_HEADS (16384 counters, 64 KB
// per device); larger calls return GDN_ERR_UNSUPPORTED before anything runs.
// All calls on one device share the one array: two calls that can run on the
// GPU at the same time (streams with no ordering between them, host threads
// racing on different streams) race on the counters and their results are
// undefined.  Calls ordered on one stream are fine.  Make the first call on
// each device before any stream capture begins, since that call does the
// symbol lookup.  Calls after cudaDeviceReset of a device are not supported
// (the cached address belongs to the old context).
#include <atomic>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.cuh"

static __device__ __align__(256) int32_t g_noalloc_counters[GDN_NOALLOC_MAX_KEY_HEADS];

namespace gdn {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int32_t *> g_counters_of[kMaxDevices];   // per device id, set once
std::mutex g_setup_mutex;

// The device address of g_noalloc_counters for the current device, looked up
// on the first call per device (with that device current) and cached for the
// life of the process.  The cache is not told about a device reset: after
// cudaDeviceReset the module is loaded again in a new context and the cached
// address is stale, so calls after a reset of that device are not supported.
cudaError_t noalloc_counters(int32_t **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int32_t *ptr = g_counters_of[dev].load(std::memory_order_acquire);
    if (ptr == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        ptr = g_counters_of[dev].load(std::memory_order_relaxed);
        if (ptr == nullptr) {
            e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_counters);
            if (e != cudaSuccess) return e;
            if (ptr == nullptr) return cudaErrorInvalidSymbol;
            g_counters_of[dev].store(ptr, std::memory_order_release);
        }
    }
    *out = ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace gdn

extern "C" {

GDN_API int gdn_decode_conv_norm_noalloc(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                         float *conv_state, int64_t conv_pitch, int taps,
                                         const float *x, const float *conv_w,
                                         const float *br, const float *ar, const float *dt, const float *rate,
                                         const float *z, const float *gn, float l2_eps, float eps,
                                         uint16_t *out,
                                         int batch, int nk, int nv, int d,
                                         int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                                         int64_t out_stride, void *stream)
{
    if (batch > 0 && nk > 0 && (int64_t)batch * nk > GDN_NOALLOC_MAX_KEY_HEADS) return GDN_ERR_UNSUPPORTED;
    // the checks of gdn_decode_conv_norm run first; the address lookup only once they pass
    return gdn::decode_conv_norm_entry(state, state_dtype, state_pitch, conv_state, conv_pitch, taps, x, conv_w,
                                       br, ar, dt, rate, z, gn, l2_eps, eps, out, nullptr, gdn::noalloc_counters,
                                       batch, nk, nv, d, x_stride, gate_stride, z_stride, out_stride, stream);
}

}  // extern "C"
