// Memory read probe: a plain streaming sum over a buffer.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch", the paragraph after the
// w4gemv timings: the card's read ceiling is measured as a plain sum over memory,
// and the GEMV is reported as a fraction of it.
//
// Result: the sum of the buffer's uint32 words mod 2^64. Integer addition is
// associative, so the per-CTA partials may be combined with atomics and the
// result is still exact and run-to-run identical.
//
// Layout: a persistent grid (a few CTAs per SM); each thread keeps 8 independent
// 128-bit streaming loads in flight per iteration.
#include "common.cuh"
#include "internal.h"

namespace w4 {

__device__ __forceinline__ unsigned long long sum4(uint4 v)
{
    return (unsigned long long)v.x + v.y + v.z + v.w;
}

__global__ void __launch_bounds__(512)
read_probe_kernel(unsigned long long *__restrict__ sum, const uint4 *__restrict__ buf,
                  long long nvec)
{
    pdl_launch_dependents();
    pdl_wait();
    constexpr int UNR = 8;
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    unsigned long long acc = 0ull;
    for (; i + (UNR - 1) * stride < nvec; i += UNR * stride) {
        uint4 v[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u)
            v[u] = ldg_stream_v4(buf + i + u * stride);
#pragma unroll
        for (int u = 0; u < UNR; ++u)
            acc += sum4(v[u]);
    }
    for (; i < nvec; i += stride)
        acc += sum4(ldg_stream_v4(buf + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    __shared__ unsigned long long ws[16];
    if ((threadIdx.x & 31) == 0)
        ws[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0ull;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            s += ws[w];
        atomicAdd(sum, s);
    }
}

cudaError_t run_read_probe(unsigned long long *sum, const void *buf, size_t bytes, int num_sms,
                           cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(sum, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess)
        return e;
    const long long nvec = (long long)(bytes / 16);
    long long blocks = (long long)num_sms * 4;
    const long long need = (nvec + 511) / 512;
    if (blocks > need)
        blocks = need;
    if (blocks < 1)
        blocks = 1;
    read_probe_kernel<<<(unsigned)blocks, 512, 0, s>>>(sum, (const uint4 *)buf, nvec);
    return cudaGetLastError();
}

} // namespace w4
