// Walsh-Hadamard transform of the activation for Hadamard-rotated W4 weights.
//
// Source: "fastgemma-gemma-4-E2B" model card, "What is in the file": every
// linear weight is Hadamard-rotated along K (W' = W H^T, H orthogonal), and a
// runtime fast Walsh-Hadamard transform of the activation makes the product
// identical while both weight groups and activation rows lose their outliers.
// H = blockdiag(H_b) over blocks of b consecutive k, H_b[i][j] =
// (-1)^popcount(i & j) / sqrt(b) (symmetric), so y = x W^T = (x H) W'^T.
//
// GB300 design. x H is computed once per call, in fp32: for blocks of 256 or
// 512 by one warp per block with the values in registers (lane exchanges for
// the upper index bits); otherwise by one CTA per (x-row, block of b) whose
// log2(b) butterfly stages run in shared memory. The result
// is split into two bf16 parts, hi = bf16(v) and lo = bf16(v - hi), so that
// |v - hi - lo| <= 2^-18 |v| (a single bf16 would cost 2^-9, far above the
// decode tolerance). The parts are written as x-rows 2m and 2m+1 of a scratch
// activation; the decode kernels run on the 2M rows and add each pair before
// storing. For M = 1 the pair fills the mma columns that a single row leaves
// empty, so the split costs no tensor work and no extra weight traffic. For
// M = 1 with blocks of 256 or 512 the decode kernel itself performs the same
// stages while it stages x (gemv_decode.cu), and this kernel is not launched.
#include "common.cuh"
#include "internal.h"

#include <cuda_bf16.h>

#include <cmath>

namespace w4 {

namespace {

__global__ void __launch_bounds__(256)
hadamard_split_kernel(uint16_t *__restrict__ x2, const uint16_t *__restrict__ x, int K, int b,
                      int lgb, float norm)
{
    extern __shared__ float v[]; // b values of one block
    pdl_launch_dependents();
    pdl_wait(); // x may be the previous kernel's output
    const int m = blockIdx.y;
    const int k0 = blockIdx.x * b;
    const uint16_t *xr = x + (size_t)m * K + k0;
    for (int i = threadIdx.x; i < b; i += blockDim.x)
        v[i] = bf16lo_to_f32(xr[i]);
    __syncthreads();
    // Stage h: pairs (j, j + h) with bit h of j clear; (p, q) -> (p + q, p - q).
    for (int s = 0; s < lgb; ++s) {
        const int h = 1 << s;
        for (int i = threadIdx.x; i < (b >> 1); i += blockDim.x) {
            const int j = ((i >> s) << (s + 1)) | (i & (h - 1));
            const float p = v[j], q = v[j + h];
            v[j] = p + q;
            v[j + h] = p - q;
        }
        __syncthreads();
    }
    uint16_t *hi = x2 + (size_t)(2 * m) * K + k0;
    uint16_t *lo = hi + K;
    for (int i = threadIdx.x; i < b; i += blockDim.x) {
        const float r = v[i] * norm;
        const __nv_bfloat16 h16 = __float2bfloat16_rn(r);
        hi[i] = __bfloat16_as_ushort(h16);
        lo[i] = __bfloat16_as_ushort(__float2bfloat16_rn(r - __bfloat162float(h16)));
    }
}

// Blocks of b = 32 * PL (PL = 8 or 16): one warp per block, lane l holding
// values [PL*l, PL*l + PL) in registers; the butterfly stages over the low
// log2(PL) index bits stay in the lane, the next five are lane exchanges
// (shfl_xor). Same stage order and pairing as the kernel above, so the same
// bits, without a CTA barrier per stage.
template <int PL>
__global__ void __launch_bounds__(128)
hadamard_split_warp_kernel(uint16_t *__restrict__ x2, const uint16_t *__restrict__ x, int K, float norm)
{
    constexpr int B = 32 * PL, NC = PL / 8;
    pdl_launch_dependents();
    pdl_wait(); // x may be the previous kernel's output
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.y;
    const int blk = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk * B >= K)
        return;
    const uint16_t *src = x + (size_t)m * K + blk * B + lane * PL;
    float v[PL];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src + 8 * c);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * c + 2 * j] = bf16lo_to_f32(u[j]);
            v[8 * c + 2 * j + 1] = bf16hi_to_f32(u[j]);
        }
    }
#pragma unroll
    for (int h = 1; h < PL; h <<= 1)
#pragma unroll
        for (int r = 0; r < PL; ++r)
            if (!(r & h)) {
                const float p = v[r], q = v[r + h];
                v[r] = p + q;
                v[r + h] = p - q;
            }
#pragma unroll
    for (int mk = 1; mk < 32; mk <<= 1) {
        const bool upper = (lane & mk) != 0;
#pragma unroll
        for (int r = 0; r < PL; ++r) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[r], mk);
            v[r] = upper ? o - v[r] : v[r] + o;
        }
    }
    uint16_t *hi = x2 + (size_t)(2 * m) * K + blk * B + lane * PL;
    uint16_t *lo = hi + K;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float r0 = v[8 * c + 2 * j] * norm, r1 = v[8 * c + 2 * j + 1] * norm;
            const __nv_bfloat16 h0 = __float2bfloat16_rn(r0), h1 = __float2bfloat16_rn(r1);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(r0 - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(r1 - __bfloat162float(h1));
            hw[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[j] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
        }
        *reinterpret_cast<uint4 *>(hi + 8 * c) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(lo + 8 * c) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

} // namespace

cudaError_t run_hadamard_split(uint16_t *x2, const uint16_t *x, int M, int K, int b, cudaStream_t s)
{
    if (b == 256 || b == 512) {
        const int nblk = K / b;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((nblk + 3) / 4, M);
        cfg.blockDim = dim3(128);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const float norm = (float)(1.0 / std::sqrt((double)b));
        return b == 256 ? cudaLaunchKernelEx(&cfg, hadamard_split_warp_kernel<8>, x2, x, K, norm)
                        : cudaLaunchKernelEx(&cfg, hadamard_split_warp_kernel<16>, x2, x, K, norm);
    }
    int lgb = 0;
    while ((1 << lgb) < b)
        ++lgb;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(K / b, M);
    cfg.blockDim = dim3(b / 2 < 256 ? (b / 2 < 32 ? 32 : b / 2) : 256);
    cfg.dynamicSmemBytes = (size_t)b * sizeof(float);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float norm = (float)(1.0 / std::sqrt((double)b));
    return cudaLaunchKernelEx(&cfg, hadamard_split_kernel, x2, x, K, b, lgb, norm);
}

} // namespace w4
