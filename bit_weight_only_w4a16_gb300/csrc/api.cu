// C ABI of libw4a16.so: argument validation, per-device set-up and dispatch.
// The declarations, with the meaning, layout, ownership and error behaviour of
// every argument, are in include/w4a16.h.
#include "../../include/w4a16.h"
#include "internal.h"

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
// Argmax scratch: one 64-bit key per (x-row, CTA); 8 rows x 65536 CTAs.
constexpr size_t kKeyCapacity = 8u * 65536u;
// Prefill split-K scratch: 8 Mi fp32 partials (32 MiB).
constexpr size_t kWsFloats = 8u << 20;

struct DeviceState {
    // Set (release) once the fields below are written; read (acquire) first.
    std::atomic<bool> ready{false};
    int num_sms = 0;
    unsigned long long *keys = nullptr;
    int *err = nullptr; // device error word written by kernels whose bounded waits ran out
    float *ws = nullptr; // prefill split-K partials
};

DeviceState g_dev[kMaxDevices];

std::mutex g_mu;
thread_local char g_cuda_err[256] = "";

int cuda_fail(cudaError_t e)
{
    std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return W4_ERR_CUDA;
}

// Set up (once) and return the state of the current device.
int device_state(DeviceState **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return W4_ERR_NO_DEVICE;
    DeviceState &st = g_dev[dev];
    if (st.ready.load(std::memory_order_acquire)) {
        *out = &st;
        return W4_OK;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return W4_ERR_NO_DEVICE;
        }
        if (major != 10 || minor != 3)
            return W4_ERR_NO_DEVICE; // kernels are built for sm_103a only
        void *p = nullptr;
        e = cudaMalloc(&p, kKeyCapacity * sizeof(unsigned long long) + 256);
        if (e != cudaSuccess)
            return cuda_fail(e);
        st.keys = static_cast<unsigned long long *>(p);
        st.err = reinterpret_cast<int *>(static_cast<char *>(p) + kKeyCapacity * sizeof(unsigned long long));
        e = cudaMemset(st.err, 0, sizeof(int));
        if (e != cudaSuccess)
            return cuda_fail(e);
        void *w = nullptr;
        e = cudaMalloc(&w, kWsFloats * sizeof(float));
        if (e != cudaSuccess)
            return cuda_fail(e);
        st.ws = static_cast<float *>(w);
        st.num_sms = sms;
        // One-time lookups that plans use, done here so that a call captured
        // into a graph later makes none of them.
        w4::tmap_encoder();
        w4::m8_cluster_capacity();
        st.ready.store(true, std::memory_order_release);
    }
    *out = &st;
    return W4_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_attn_args(const float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const int32_t *kpos, int window, int H, int T, int D)
{
    if (!out || !q || !k || !v)
        return W4_ERR_INVALID_ARG;
    if (H < 1 || T < 1 || D < 1 || window < 0)
        return W4_ERR_INVALID_ARG;
    if (H > 8 || D % 128 != 0 || D > 512)
        return W4_ERR_UNSUPPORTED;
    if ((long long)T * D >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 4) ||
        (kpos && !aligned(kpos, 4)))
        return W4_ERR_MISALIGNED;
    return W4_OK;
}

int check_w4_args(const void *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int M,
                  int N, int K, int group)
{
    if (!y || !x || !qw || !sc)
        return W4_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0)
        return W4_ERR_INVALID_ARG;
    if (w4::group_shift(group) < 0)
        return W4_ERR_UNSUPPORTED;
    if (K % group != 0)
        return W4_ERR_INVALID_ARG;
    // Every flat index the kernels form stays below 2^31 words or elements.
    if ((long long)N * (K / 8) >= (1ll << 31) || (long long)M * K >= (1ll << 31) ||
        (long long)M * N >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qw, 16) || !aligned(sc, 4) || !aligned(y, 4))
        return W4_ERR_MISALIGNED;
    return W4_OK;
}

// Shared memory the decode kernels need for x staging; bounded by the SM's 227 KB.
bool decode_fits(const w4::DecodePlan &p, int M, int K)
{
    return w4::decode_smem_bytes(p, M, K) <= 220 * 1024;
}

} // namespace

extern "C" {

const char *w4_status_string(int status)
{
    switch (status) {
    case W4_OK: return "W4_OK";
    case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG";
    case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED";
    case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED";
    case W4_ERR_CUDA: return "W4_ERR_CUDA";
    case W4_ERR_NO_DEVICE: return "W4_ERR_NO_DEVICE";
    default: return "W4_ERR_UNKNOWN";
    }
}

const char *w4_last_cuda_error(void) { return g_cuda_err; }

int w4_init(void)
{
    DeviceState *st = nullptr;
    return device_state(&st);
}

int w4a16_gemv(float *y, const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, int M,
               int N, int K, int group, void *stream)
{
    int rc = check_w4_args(y, x, qweight, scales, M, N, K, group);
    if (rc != W4_OK)
        return rc;
    if (M > 8)
        return W4_ERR_UNSUPPORTED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int lg = w4::group_shift(group);
    if (w4::vocab_supported(M, N, K, st->num_sms, lg, qweight, scales)) {
        cudaError_t e = w4::run_decode_vocab(y, x, qweight, scales, N, K, lg, nullptr, nullptr, st->err,
                                             st->num_sms, s);
        return e == cudaSuccess ? W4_OK : cuda_fail(e);
    }
    if (M == 1) {
        // Measured on GB300 in the graph-replayed sweep: the slot form first
        // (0.505 -> 0.473 ms; 1536 x 6144 3.56 -> 3.29 us, 2560 x 1536 2.23 ->
        // 2.19 us), the few-tiles-per-warp form for the shapes it cannot take
        // (K % 768 != 0: 1536 x 2048).
        const int R = w4::slab_rows_per_cta(M, N, K, st->num_sms, lg, qweight, scales);
        if (R > 0) {
            cudaError_t e = w4::run_decode_slab(R, y, x, qweight, scales, N, K, st->err, s);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
        const w4::M1Plan mp = w4::plan_decode_m1(M, N, K, st->num_sms);
        if (mp.ok) {
            cudaError_t e = w4::run_decode_m1(mp, y, x, qweight, scales, N, K, lg, s);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
    } else {
        const w4::Slots8Plan sp = w4::plan_slots8(M, N, K, st->num_sms, lg, qweight, scales);
        if (sp.ok) {
            cudaError_t e = w4::run_decode_slots8(sp, y, x, qweight, scales, M, N, K, nullptr, nullptr, st->err, s);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
    }
    const w4::DecodePlan p = w4::plan_decode(M, N, K, st->num_sms);
    if (!decode_fits(p, M, K))
        return W4_ERR_UNSUPPORTED;
    cudaError_t e = w4::run_decode(p, y, x, qweight, scales, M, N, K, lg, nullptr, nullptr, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4a16_gemm(float *y, const uint16_t *x, const uint32_t *qweight, const uint16_t *scales, int M,
               int N, int K, int group, void *stream)
{
    if (M >= 1 && M <= 8)
        return w4a16_gemv(y, x, qweight, scales, M, N, K, group, stream);
    int rc = check_w4_args(y, x, qweight, scales, M, N, K, group);
    if (rc != W4_OK)
        return rc;
    if (N % 16 != 0 || K % 64 != 0)
        return W4_ERR_UNSUPPORTED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    const w4::PrefillPlan p = w4::plan_prefill(M, N, K, st->num_sms, kWsFloats);
    cudaError_t e = w4::run_prefill(p, y, x, qweight, scales, M, N, K, w4::group_shift(group), st->ws, st->err,
                                    static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported)
        return W4_ERR_UNSUPPORTED;
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4a16_gemv_argmax(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                      const uint16_t *scales, int M, int N, int K, int group, void *stream)
{
    int rc = check_w4_args(y, x, qweight, scales, M, N, K, group);
    if (rc != W4_OK)
        return rc;
    if (!argmax)
        return W4_ERR_INVALID_ARG;
    if (!aligned(argmax, 4))
        return W4_ERR_MISALIGNED;
    if (M > 8)
        return W4_ERR_UNSUPPORTED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int lg = w4::group_shift(group);
    if (w4::vocab_supported(M, N, K, st->num_sms, lg, qweight, scales)) {
        cudaError_t e = w4::run_decode_vocab(y, x, qweight, scales, N, K, lg, st->keys, argmax, st->err,
                                             st->num_sms, s);
        return e == cudaSuccess ? W4_OK : cuda_fail(e);
    }
    if (M >= 2) {
        const w4::Slots8Plan sp = w4::plan_slots8(M, N, K, st->num_sms, lg, qweight, scales);
        if (sp.ok && (size_t)M * sp.grid <= kKeyCapacity) {
            cudaError_t e = w4::run_decode_slots8(sp, y, x, qweight, scales, M, N, K, st->keys, argmax, st->err, s);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
    }
    const w4::DecodePlan p = w4::plan_decode(M, N, K, st->num_sms);
    if (!decode_fits(p, M, K) || (size_t)M * p.grid > kKeyCapacity)
        return W4_ERR_UNSUPPORTED;
    cudaError_t e = w4::run_decode(p, y, x, qweight, scales, M, N, K, lg, st->keys, argmax, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_embed_gather(uint16_t *out, const int32_t *ids, const uint32_t *qtable,
                    const uint16_t *scales, int M, int N, int K, int group, int32_t *status,
                    void *stream)
{
    if (!out || !ids || !qtable || !scales)
        return W4_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0)
        return W4_ERR_INVALID_ARG;
    if (w4::group_shift(group) < 0)
        return W4_ERR_UNSUPPORTED;
    if (K % group != 0)
        return W4_ERR_INVALID_ARG;
    if ((long long)N * (K / 8) >= (1ll << 31) || (long long)M * K >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(qtable, 4) || !aligned(scales, 2) || !aligned(ids, 4) ||
        (status && !aligned(status, 4)))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = w4::run_embed_gather(out, ids, qtable, scales, M, N, K, w4::group_shift(group), status,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_device_error(int32_t *code)
{
    if (!code)
        return W4_ERR_INVALID_ARG;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(code, st->err, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemset(st->err, 0, sizeof(int32_t));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int hbm_read_probe(unsigned long long *sum, const void *buf, size_t bytes, void *stream)
{
    if (!sum || !buf || bytes == 0)
        return W4_ERR_INVALID_ARG;
    if (bytes % 16 != 0)
        return W4_ERR_INVALID_ARG;
    if (!aligned(buf, 16) || !aligned(sum, 8))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = w4::run_read_probe(sum, buf, bytes, st->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_attn_decode(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *kpos, int qpos, int window, int H, int T, int D, float scale,
                   void *stream)
{
    int rc = check_attn_args(out, q, k, v, kpos, window, H, T, D);
    if (rc != W4_OK)
        return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    cudaError_t e = w4::run_attn_decode(out, q, k, v, kpos, qpos, nullptr, window, H, T, D, scale, st->ws,
                                        kWsFloats, st->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4a16_gemv_hadamard(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, int M, int N, int K, int group, int hblock, void *stream)
{
    int rc = check_w4_args(y, x, qweight, scales, M, N, K, group);
    if (rc != W4_OK)
        return rc;
    if (hblock < 2 || hblock > 4096 || (hblock & (hblock - 1)) != 0)
        return W4_ERR_UNSUPPORTED;
    if (K % hblock != 0)
        return W4_ERR_INVALID_ARG;
    if (M > 4)
        return W4_ERR_UNSUPPORTED;
    if (argmax && !aligned(argmax, 4))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // One x-row, blocks of 256 or 512, K % 128 == 0, the shared-memory slot
    // form or the M <= 2 kernel (not the large-N forms, where the separate
    // transform overlaps the weight preload and measured faster): the decode
    // kernel forms x H itself while staging x (no transform launch, no scratch
    // rows).
    if (M == 1 && !argmax) {
        const int R = w4::slab_rows_per_cta(M, N, K, st->num_sms, w4::group_shift(group), qweight, scales, hblock);
        if (R > 0) {
            cudaError_t e = w4::run_decode_slab(R, y, x, qweight, scales, N, K, st->err, s, hblock);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
    }
    if (M == 1 && (hblock == 256 || hblock == 512) && K % 128 == 0) {
        const w4::DecodePlan p = w4::plan_decode(2, N, K, st->num_sms);
        if (p.kernel == 2 && decode_fits(p, 2, K) && (!argmax || (size_t)p.grid <= kKeyCapacity)) {
            cudaError_t e = w4::run_decode(p, y, x, qweight, scales, 2, N, K, w4::group_shift(group),
                                           argmax ? st->keys : nullptr, argmax, s, true, nullptr, hblock);
            return e == cudaSuccess ? W4_OK : cuda_fail(e);
        }
    }
    // The rotated activation's (hi, lo) rows live in the split scratch.
    if ((size_t)2 * M * K * sizeof(uint16_t) > kWsFloats * sizeof(float))
        return W4_ERR_UNSUPPORTED;
    const w4::DecodePlan p = w4::plan_decode(2 * M, N, K, st->num_sms);
    if (!decode_fits(p, 2 * M, K) || (argmax && (size_t)M * p.grid > kKeyCapacity))
        return W4_ERR_UNSUPPORTED;
    uint16_t *x2 = reinterpret_cast<uint16_t *>(st->ws);
    cudaError_t e = w4::run_hadamard_split(x2, x, M, K, hblock, s);
    if (e == cudaSuccess)
        e = w4::run_decode(p, y, x2, qweight, scales, 2 * M, N, K, w4::group_shift(group),
                           argmax ? st->keys : nullptr, argmax, s, true);
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_selftest_wait_timeout(void *stream)
{
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = w4::run_bounded_wait_selftest(st->err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_attn_decode_devpos(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *kpos, const int32_t *qpos, int window, int H, int T, int D,
                          float scale, void *stream)
{
    int rc = check_attn_args(out, q, k, v, kpos, window, H, T, D);
    if (rc != W4_OK)
        return rc;
    if (!qpos)
        return W4_ERR_INVALID_ARG;
    if (!aligned(qpos, 4))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    cudaError_t e = w4::run_attn_decode(out, q, k, v, kpos, 0, qpos, window, H, T, D, scale, st->ws, kWsFloats,
                                        st->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_kv_append(uint16_t *k_cache, uint16_t *v_cache, int32_t *kpos, const uint16_t *k_new,
                 const uint16_t *v_new, const int32_t *pos, int T, int D, int32_t *status, void *stream)
{
    if (!k_cache || !v_cache || !k_new || !v_new || !pos)
        return W4_ERR_INVALID_ARG;
    if (T < 1 || D < 8 || D % 8 != 0 || (long long)T * D >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(pos, 4) || (kpos && !aligned(kpos, 4)) || (status && !aligned(status, 4)))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = w4::run_kv_append(k_cache, v_cache, kpos, k_new, v_new, pos, T, D, status,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4a16_gemv_argmax_forced(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                             const uint16_t *scales, int N, int K, int group, const int32_t *forced,
                             void *stream)
{
    int rc = check_w4_args(y, x, qweight, scales, 1, N, K, group);
    if (rc != W4_OK)
        return rc;
    if (!argmax || !forced)
        return W4_ERR_INVALID_ARG;
    if (!aligned(argmax, 4) || !aligned(forced, 4))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != W4_OK)
        return rc;
    const int lg = w4::group_shift(group);
    if (w4::vocab_supported(1, N, K, st->num_sms, lg, qweight, scales)) {
        cudaError_t e = w4::run_decode_vocab(y, x, qweight, scales, N, K, lg, st->keys, argmax, st->err,
                                             st->num_sms, static_cast<cudaStream_t>(stream), forced);
        return e == cudaSuccess ? W4_OK : cuda_fail(e);
    }
    const w4::DecodePlan p = w4::plan_decode(1, N, K, st->num_sms);
    if (p.kernel == 8 || !decode_fits(p, 1, K) || (size_t)p.grid > kKeyCapacity)
        return W4_ERR_UNSUPPORTED;
    cudaError_t e = w4::run_decode(p, y, x, qweight, scales, 1, N, K, w4::group_shift(group), st->keys, argmax,
                                   static_cast<cudaStream_t>(stream), false, forced);
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

int w4_decode_prologue(uint16_t *x_next, int32_t *tokens, int32_t *pos, const int32_t *token,
                       const uint32_t *qtable, const uint16_t *scales, int V, int K, int group, int cap,
                       int32_t *status, void *stream)
{
    if (!x_next || !pos || !token || !qtable || !scales)
        return W4_ERR_INVALID_ARG;
    if (V < 1 || K < 1 || (tokens && cap < 1))
        return W4_ERR_INVALID_ARG;
    if (w4::group_shift(group) < 0)
        return W4_ERR_UNSUPPORTED;
    if (K % group != 0 || (long long)V * (K / 8) >= (1ll << 31))
        return W4_ERR_INVALID_ARG;
    if (!aligned(x_next, 16) || !aligned(qtable, 4) || !aligned(scales, 2) || !aligned(pos, 4) ||
        !aligned(token, 4) || (tokens && !aligned(tokens, 4)) || (status && !aligned(status, 4)))
        return W4_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != W4_OK)
        return rc;
    cudaError_t e = w4::run_decode_prologue(x_next, tokens, pos, token, qtable, scales, V, K,
                                            w4::group_shift(group), tokens ? cap : 0, status,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4_OK : cuda_fail(e);
}

} // extern "C"
