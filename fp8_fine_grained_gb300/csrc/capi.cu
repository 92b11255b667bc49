// Status word, device queries and diagnostics of libfp8fg.so.
#include <atomic>
#include <mutex>

#include "host_common.h"

namespace {

// Per-device status word. Kernels record the first device-side error with
// atomicCAS(…, 0, code); fp8fg_device_status reads and clears it.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceCache {
    std::once_flag once;
    int *status = nullptr;
    int sms = 0;
    bool supported = false;
};

DeviceCache g_dev[kMaxDevices];
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_skinny_rows{32};
std::atomic<int> g_skinny_cost_pct{100};
std::atomic<int> g_skip_first_load[kMaxDevices];

DeviceCache *cache_for_current()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    DeviceCache *c = &g_dev[dev];
    std::call_once(c->once, [c, dev]() {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess)
            c->status = static_cast<int *>(p);
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            c->sms = v;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        c->supported = (major == 10 && minor == 3);
        cudaGetLastError();
    });
    return c;
}

}  // namespace

namespace fp8fg {

int *status_word_ptr()
{
    DeviceCache *c = cache_for_current();
    return c ? c->status : nullptr;
}

int sm_count()
{
    DeviceCache *c = cache_for_current();
    return c ? c->sms : 0;
}

bool device_supported()
{
    DeviceCache *c = cache_for_current();
    return c && c->supported && c->status != nullptr;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

int grouped_skinny_rows() { return g_skinny_rows.load(); }

int grouped_skinny_cost_pct() { return g_skinny_cost_pct.load(); }

bool take_skip_first_load()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return false;
    return g_skip_first_load[dev].exchange(0) != 0;
}

}  // namespace fp8fg

extern "C" {

const char *fp8fg_status_str(int status)
{
    switch (status) {
    case FP8FG_OK: return "FP8FG_OK";
    case FP8FG_EINVAL: return "FP8FG_EINVAL: invalid argument";
    case FP8FG_EALIGN: return "FP8FG_EALIGN: pointer or pitch not 16-byte aligned";
    case FP8FG_EUNSUPPORTED: return "FP8FG_EUNSUPPORTED: device is not sm_103";
    case FP8FG_ECUDA: return "FP8FG_ECUDA: CUDA error";
    case FP8FG_ETIMEOUT: return "FP8FG_ETIMEOUT: a device-side bounded wait ran out";
    case FP8FG_EDEVICE: return "FP8FG_EDEVICE: invalid data found on the device";
    default: return "FP8FG: unknown status";
    }
}

int fp8fg_device_status(void *stream)
{
    int *p = fp8fg::status_word_ptr();
    if (!p)
        return FP8FG_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return FP8FG_ECUDA;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8FG_ECUDA;
    if (v != 0) {
        int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8FG_ECUDA;
    }
    return v;
}

int fp8fg_version(void) { return 100; }

int fp8fg_test_skip_first_load(int skip)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    g_skip_first_load[dev].store(skip ? 1 : 0);
    return FP8FG_OK;
}

int fp8fg_set_wait_limit_ns(int64_t ns)
{
    if (ns < 1000000)
        ns = 1000000;
    g_wait_limit_ns.store(static_cast<uint64_t>(ns));
    return FP8FG_OK;
}

int fp8fg_set_grouped_schedule(int skinny_rows, int skinny_cost_pct)
{
    if (skinny_rows < 0 || skinny_rows > 32 || skinny_cost_pct < 1 || skinny_cost_pct > 1000)
        return FP8FG_EINVAL;
    g_skinny_rows.store(skinny_rows);
    g_skinny_cost_pct.store(skinny_cost_pct);
    return FP8FG_OK;
}

}  // extern "C"
