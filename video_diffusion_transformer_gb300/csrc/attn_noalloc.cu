// fv_attn_fwd_noalloc: the attention entry point for callers that must not
// allocate device memory.
//
// fv_attn_fwd keeps a small device status word that the library allocates
// with cudaMalloc the first time it runs on a device.  Some callers cannot let
// a library do that: their device memory belongs to someone else (a
// framework's caching allocator, or a serving process with a fixed memory
// budget that accounts for every byte), and cudaMalloc may also synchronise
// the whole device at a moment the caller does not control.  This variant
// runs the same attention kernel but keeps its scratch -- one status word per
// head-group launch -- in a fixed array compiled into the library.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fv.h"
#include "fv_internal.h"

// The scratch: one status word per head-group launch of a call, so at most
// FV_NOALLOC_MAX_LAUNCHES launches (256 bytes).  Every GPU that loads the
// library holds this array until the process exits.  Host code must not use
// the name as an address; it asks the runtime for the device address below.
static __device__ __align__(256) int g_noalloc_status[FV_NOALLOC_MAX_LAUNCHES];

namespace {

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int *status = nullptr;  // device address of g_noalloc_status on this device
};

std::mutex g_mu;
NoAllocDevice g_devs[kMaxDevices];

// Once per device, with that device current: check the architecture, count
// the SMs and look up the device address of the scratch array.  Nothing here
// allocates.
fv_status setup_current_device(NoAllocDevice **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FV_ERR_LAUNCH;
    std::lock_guard<std::mutex> g(g_mu);
    NoAllocDevice &d = g_devs[dev];
    if (!d.ready) {
        if (!fv::probe_device(dev, &d.supported, &d.num_sms)) return FV_ERR_LAUNCH;
        if (d.supported) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_status) != cudaSuccess || p == nullptr) return FV_ERR_LAUNCH;
            d.status = static_cast<int *>(p);
        }
        d.ready = true;
    }
    if (!d.supported) return FV_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return FV_OK;
}

}  // namespace

extern "C" fv_status fv_attn_fwd_noalloc(const void *Q, const void *K, const void *V, void *O, int64_t N, int H,
                                         int D, float scale, int head_group, float *lse, void *stream,
                                         int *device_status_out) {
    fv::NvtxRange nvtx("fv_attn_fwd_noalloc");
    // the same checks as fv_attn_fwd, then the scratch limit
    fv_status st = fv::check_attn_args(Q, K, V, O, N, H, D, scale, head_group, lse);
    if (st != FV_OK) return st;
    const int launches = (H + head_group - 1) / head_group;
    if (launches > FV_NOALLOC_MAX_LAUNCHES) return FV_ERR_SHAPE;  // more launches than scratch words
    NoAllocDevice *d = nullptr;
    st = setup_current_device(&d);
    if (st != FV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's words: clear the ones this call uses.
    if (cudaMemsetAsync(d->status, 0, sizeof(int) * (size_t)launches, s) != cudaSuccess) return FV_ERR_LAUNCH;
    fv::AttnLaunch a;
    a.q = Q;
    a.k = K;
    a.v = V;
    a.o = O;
    a.lse = lse;
    a.n = N;
    a.heads_total = H;
    a.scale = scale;
    a.num_sms = d->num_sms;
    for (int i = 0; i < launches; ++i) {
        a.head_begin = i * head_group;
        a.heads = (H - a.head_begin) < head_group ? (H - a.head_begin) : head_group;
        a.status = d->status + i;
        st = fv::launch_attn_fwd(a, s);
        if (st != FV_OK) return st;
    }
    if (device_status_out != nullptr) {
        int words[FV_NOALLOC_MAX_LAUNCHES] = {0};
        if (cudaMemcpyAsync(words, d->status, sizeof(int) * (size_t)launches, cudaMemcpyDeviceToHost, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return FV_ERR_LAUNCH;
        fv_status dev_st = FV_OK;
        for (int i = 0; i < launches; ++i)
            if (words[i] != 0 && dev_st == FV_OK) dev_st = fv::status_of_word(words[i]);
        *device_status_out = (int)dev_st;
    }
    return FV_OK;
}
