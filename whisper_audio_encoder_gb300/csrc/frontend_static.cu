// wh_frontend_static: the log-mel front end for callers that cannot allocate device memory.
//
// wh_frontend needs a small caller-provided scratch buffer (one word per window for the
// window's maximum log-mel value, one for the kernel's grid barrier).  Some callers have no way to provide one at the point
// they call in: a real-time audio callback must not block on the CUDA allocator
// (cudaMalloc can synchronise the device and take milliseconds), and a process that has
// handed all of its device memory to another allocator up front has none left to give.
// This entry point keeps that scratch in a fixed array inside the library instead, so it
// allocates nothing: the caller still passes the PCM input and the log-mel output.
//
// The array below is a file-scope device variable: every GPU that loads the library holds
// its WH_FRONTEND_STATIC_MAX_BATCH + 1 words until the process exits.  Host code cannot use the
// name of a device variable as an address (on the host it names a host-side stand-in), so
// the device address is looked up once per device with cudaGetSymbolAddress and passed to
// the kernels.  All calls on a device share the one array, so calls that overlap on the GPU
// (two streams at once) race on it; the per-window maxima are cleared at the start of every
// call, so nothing carries over from the previous call.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace wh {
namespace {

static __device__ __align__(256) uint32_t g_frontend_scratch[WH_FRONTEND_STATIC_MAX_BATCH + 1];

constexpr int MAX_DEV = 64;
uint32_t *g_scratch_ptr[MAX_DEV] = {};
std::mutex g_scratch_mu;

// Once per device, with that device current: the library's own tables, then the device
// address of the scratch array.
int scratch_for_current_device(uint32_t **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) {
        cudaGetLastError();
        return WH_ENODEV;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        if (int rc = device_setup()) return rc;
        uint32_t *p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_frontend_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return WH_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return WH_OK;
}

}  // namespace
}  // namespace wh

extern "C" int wh_frontend_static(const float *pcm, int64_t n, int batch, int n_mels, float *mel, void *stream) {
    using namespace wh;
    if (batch < 0 || n < 0 || (n_mels != 80 && n_mels != 128)) return WH_EINVAL;
    if (batch > WH_FRONTEND_STATIC_MAX_BATCH) return WH_ENOSPC;
    if (batch == 0) return WH_OK;
    if (!mel || (n > 0 && !pcm) || (reinterpret_cast<uintptr_t>(mel) % 16) != 0) return WH_EINVAL;
    uint32_t *scratch = nullptr;
    if (int rc = scratch_for_current_device(&scratch)) return rc;
    DevCtl ctl;
    int num_sms = 0;
    if (int rc = frontend_ctl(&ctl, &num_sms)) return rc;
    // frontend_launch clears the per-window maxima and the barrier count (cudaMemsetAsync)
    // before its kernel runs.
    return frontend_launch(pcm, n, n, n * batch, batch, n_mels, mel, scratch, ctl, num_sms,
                           static_cast<cudaStream_t>(stream));
}
