// A stage-2 step for callers that cannot allocate device memory.
//
// The regular step needs two pieces of scratch besides the caller's model
// buffers: a 4 KB workspace (overflow flag, exact sum-of-squares
// accumulators, norm, clip coefficient) and, on the two-pass path, the
// reduced 16-bit gradient.  Some callers have no way to provide them: code
// that runs inside another runtime which owns the device's memory pool and
// hands out no allocations, or code that must not call cudaMalloc after its
// start-up phase.  zero_step_stage2_noalloc takes that scratch from one
// static device array compiled into this library instead.
//
// The array's size is fixed (see kNoAllocScratchBytes below); every GPU that
// loads the library keeps it for the life of the process.  All calls share
// it, so two calls whose kernels overlap on the GPU (different streams,
// different host threads) race on it; calls on one stream are ordered and
// safe.
#include <cstdio>
#include <mutex>

#include "zero_internal.h"

namespace {

constexpr int64_t kNoAllocMaxReduced = int64_t(8) << 20;   // 16-bit elements of the reduced gradient
constexpr size_t kNoAllocScratchBytes = zg::ws::kBytes + kNoAllocMaxReduced * 2;   // 4 KB + 16 MiB
constexpr int kMaxDevices = 64;

// In host code `g_noalloc_scratch` names a host-side stand-in for the
// symbol, not the device memory: kernels must be given the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the static scratch on device `dev` (the current device),
// looked up once per device (the first call on a device does this set-up).
cudaError_t scratch_address(int dev, void** out)
{
    cudaError_t e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" zero_status_t zero_step_stage2_noalloc(const zero_config_t* cfg, const zero_plan_t* plan,
                                                  zero_buffers_t* bufs, const zero_adam_t* adam, zero_state_t* state,
                                                  void* stream, zero_step_result_t* out)
{
    if (!cfg || !plan || !bufs)
        return zg::set_error(ZERO_EINVAL, "zero_step_stage2_noalloc: config, plan and buffers must not be NULL");
    zero_plan_t fresh;
    zero_status_t st = zero_plan(cfg, &fresh);   // checks the config, sets the error text
    if (st != ZERO_OK) return st;
    char msg[256];
    if (cfg->stage != 2) {
        std::snprintf(msg, sizeof msg, "zero_step_stage2_noalloc needs a stage-2 config (got stage %d)", cfg->stage);
        return zg::set_error(ZERO_EINVAL, msg);
    }
    if (cfg->dtype == ZERO_FP32)
        return zg::set_error(ZERO_EUNSUPPORTED, "zero_step_stage2_noalloc takes 16-bit gradients only");
    if (fresh.padded_elems > kNoAllocMaxReduced) {
        std::snprintf(msg, sizeof msg,
                      "zero_step_stage2_noalloc: the plan's padded_elems %lld exceed the %lld that fit the static "
                      "scratch (16 MiB of reduced gradient)",
                      (long long)fresh.padded_elems, (long long)kNoAllocMaxReduced);
        return zg::set_error(ZERO_EUNSUPPORTED, msg);
    }
    // The scratch address belongs to the current device, and the kernels run
    // on `stream`: both must be the same GPU.
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "zero_step_stage2_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return zg::set_error(ZERO_ECUDA, msg);
    }
    if (stream) {
        int sdev = -1;
        e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
        if (e != cudaSuccess) {
            std::snprintf(msg, sizeof msg, "zero_step_stage2_noalloc: cudaStreamGetDevice: %s",
                          cudaGetErrorString(e));
            return zg::set_error(ZERO_ECUDA, msg);
        }
        if (sdev != dev) {
            std::snprintf(msg, sizeof msg,
                          "zero_step_stage2_noalloc: the stream belongs to device %d, the current device is %d "
                          "(make the stream's device current)", sdev, dev);
            return zg::set_error(ZERO_EINVAL, msg);
        }
    }
    void* scratch = nullptr;
    e = scratch_address(dev, &scratch);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "zero_step_stage2_noalloc: cudaGetSymbolAddress of the static scratch: %s",
                      cudaGetErrorString(e));
        return zg::set_error(ZERO_ECUDA, msg);
    }
    // The regular stage-2 step with the scratch pointed at the static array:
    // no shadow state, so the two-pass path runs and updates [cur] in place;
    // its first action clears the workspace part of the array.
    zero_buffers_t b = *bufs;
    const int sh = 1 - b.cur;
    if (sh == 0 || sh == 1) {
        b.w[sh] = nullptr;
        b.m[sh] = nullptr;
        b.v[sh] = nullptr;
    }
    b.workspace = scratch;
    b.reduced = static_cast<unsigned char*>(scratch) + zg::ws::kBytes;
    st = zero_step_stage2(cfg, plan, &b, adam, state, stream, out);
    bufs->cur = b.cur;
    return st;
}
