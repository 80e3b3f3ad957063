// Decode GEMV with the fused greedy pick that allocates no device memory.
//
// Some callers cannot call cudaMalloc at all: plug-ins loaded into a host
// process that owns every device allocation through its own allocator, and
// real-time decode loops that must not hit the driver's allocator after
// start-up. For them this entry point
// keeps its scratch (one 64-bit argmax key per CTA and x-row) in a fixed array
// in the library's own device image instead of the scratch that w4_init
// allocates.
//
// The array is a file-scope static __device__ variable: every GPU that loads
// the library holds it (256 KiB) until the process exits. Host code may not
// use its name as a device address, so the address is looked up once per device
// with cudaGetSymbolAddress, with that device current, by the first call on the
// device. Every CTA writes its key slot before the finalize kernel reads it, so
// nothing has to start at zero, but all calls share the one array: two calls
// whose kernels overlap in time on the GPU (different streams) race on it.
#include "../../include/w4a16.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace {

constexpr int kNoallocKeys = 8 * 4096; // M * CTAs of one call, at most
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned long long g_noalloc_keys[kNoallocKeys];

struct NoallocDevice {
    // Set (release) after keys and num_sms are written; read (acquire) before
    // they are used, so a concurrent first call never sees a half-made state.
    std::atomic<bool> ready{false};
    int num_sms = 0;
    unsigned long long *keys = nullptr; // device address of g_noalloc_keys
};

NoallocDevice g_na[kMaxDevices];
std::mutex g_na_mu;

// Per-device set-up, made by the first call on the device (it must come before
// any stream capture that contains this call): checks the device and resolves
// the scratch array's device address. No allocation.
int noalloc_device(NoallocDevice **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return W4_ERR_NO_DEVICE;
    }
    NoallocDevice &d = g_na[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_na_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                return W4_ERR_NO_DEVICE;
            }
            if (major != 10 || minor != 3)
                return W4_ERR_NO_DEVICE;
            unsigned long long *ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_keys);
            if (e != cudaSuccess || ptr == nullptr) {
                cudaGetLastError();
                return W4_ERR_CUDA;
            }
            d.keys = ptr;
            d.num_sms = sms;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return W4_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

} // namespace

extern "C" int w4a16_gemv_argmax_noalloc(float *y, int32_t *argmax, const uint16_t *x,
                                         const uint32_t *qweight, const uint16_t *scales, int M,
                                         int N, int K, int group, void *stream)
{
    if (!y || !argmax || !x || !qweight || !scales)
        return W4_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0)
        return W4_ERR_INVALID_ARG;
    const int lg = w4::group_shift(group);
    if (lg < 0)
        return W4_ERR_UNSUPPORTED;
    if (K % group != 0)
        return W4_ERR_INVALID_ARG;
    if ((long long)N * (K / 8) >= (1ll << 31) || (long long)M * K >= (1ll << 31) ||
        (long long)M * N >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qweight, 16) || !aligned(scales, 4) || !aligned(y, 4) ||
        !aligned(argmax, 4))
        return W4_ERR_MISALIGNED;
    if (M > 8)
        return W4_ERR_UNSUPPORTED;
    NoallocDevice *d = nullptr;
    int rc = noalloc_device(&d);
    if (rc != W4_OK)
        return rc;
    const w4::DecodePlan p = w4::plan_decode(M, N, K, d->num_sms);
    // Beyond the fixed scratch: one key per (x-row, CTA).
    if ((long long)M * p.grid > kNoallocKeys)
        return W4_ERR_UNSUPPORTED;
    if (w4::decode_smem_bytes(p, M, K) > 220 * 1024)
        return W4_ERR_UNSUPPORTED;
    const cudaError_t e = w4::run_decode(p, y, x, qweight, scales, M, N, K, lg, d->keys, argmax,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4_ERR_CUDA;
    }
    return W4_OK;
}
