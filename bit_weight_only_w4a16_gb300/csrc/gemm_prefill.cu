// Prefill W4A16 GEMM (M > 8 tokens) on the 5th-generation tensor cores.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the prompt-read
// paragraph (a prompt is read in 256-token chunks, every weight multiplies the
// whole chunk) and the Colab paragraph (on a GPU with tensor cores, 16-bit
// prompt reads run ten times faster). The pages unpack each weight matrix to a
// full 16-bit copy in memory and call a library GEMM; here the 4-bit tiles are
// dequantized on their way into shared memory and never exist as a 16-bit copy
// in HBM.
//
// y[m][n] = sum_k x[m][k] * bf16_rne((code(n,k) - 8) * step(n, k/32)), fp32
// accumulate. Rounding each weight to bf16 (relative error <= 2^-9) keeps the
// result within 2e-3 * sum|w x|.
//
// Tile: 128 weight rows (the MMA's M, TMEM lanes) x 256 tokens (the MMA's N,
// TMEM columns) x 64 k per stage (one 128-byte swizzle row of bf16), 4 stages.
//   warp 0    : TMA of the x tile (256 tokens x 64 k, 128-byte swizzle), the B operand
//   warp 1    : allocates 256 TMEM columns; lane 0 issues tcgen05.mma (4 x K=16 per
//               stage) and commits each stage's slot back to the producers
//   warps 2-5 : one thread per weight row: load 8 code words + 2 steps, dequantize
//               to bf16 and store the A tile in the K-major 128-byte-swizzle layout
//               the MMA reads; then the epilogue: tcgen05.ld of their 32 TMEM
//               lanes and coalesced fp32 stores of y.
// Every wait is bounded; a timeout sets the device error word and the kernel
// still drains its copies and MMAs and frees TMEM before returning.
#include "common.cuh"
#include "internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace w4 {

namespace {

constexpr int kBM = 128;  // weight rows per tile
constexpr int kBN = 256;  // tokens per tile
constexpr int kBK = 64;   // k per stage
constexpr int kStages = 4;
constexpr int kASlot = kBM * kBK * 2; // 16 KiB
constexpr int kBSlot = kBN * kBK * 2; // 32 KiB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr int kWait = 1 << 16;
constexpr int kDrain = 64;
constexpr size_t kSmem = (size_t)kStages * (kASlot + kBSlot) + 1024;

// tcgen05 instruction descriptor, kind::f16: fp32 D, bf16 A and B, both
// K-major, N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

// Shared-memory matrix descriptor: K-major operand in the 128-byte-swizzle
// layout (8-row x 128-byte atoms, 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout): 16 B
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
                 "l"(map), "r"(c0), "r"(c1), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// Eight codes (one word, k = 8j .. 8j+7 in order) -> eight bf16 of (code-8)*step,
// each rounded once to nearest even, as four bf16x2 in k order.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t step2, uint32_t &p01, uint32_t &p23,
                                             uint32_t &p45, uint32_t &p67)
{
    const uint32_t lo = w & 0x0F0F0F0Fu;         // codes k0 k2 k4 k6 in bytes 0..3
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes k1 k3 k5 k7
    const uint32_t m0 = __byte_perm(lo, hi, 0x5140); // k0 k1 k2 k3
    const uint32_t m1 = __byte_perm(lo, hi, 0x7362); // k4 k5 k6 k7
    // 0x43 high bytes: bf16 of 128 + code
    uint32_t q01 = __byte_perm(m0, 0x43434343u, 0x4140), q23 = __byte_perm(m0, 0x43434343u, 0x4342);
    uint32_t q45 = __byte_perm(m1, 0x43434343u, 0x4140), q67 = __byte_perm(m1, 0x43434343u, 0x4342);
    const uint32_t c136 = 0x43084308u;
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(q01) : "r"(c136));
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(q23) : "r"(c136));
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(q45) : "r"(c136));
    asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(q67) : "r"(c136));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p01) : "r"(q01), "r"(step2));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p23) : "r"(q23), "r"(step2));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p45) : "r"(q45), "r"(step2));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(p67) : "r"(q67), "r"(step2));
}

struct PrefillArgs {
    float *y;
    const uint32_t *qw;
    const uint16_t *sc;
    int *err;
    int M, N, K;
};

__global__ void __launch_bounds__(kThreads, 1)
gemm_prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap xmap)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full_a[kStages], full_b[kStages], empty[kStages];
    __shared__ __align__(8) unsigned long long acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t a_ring = smem_addr(smem);
    const uint32_t b_ring = a_ring + kStages * kASlot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBM;  // first weight row of the tile
    const int m0 = blockIdx.y * kBN;  // first token of the tile
    const int nst = a.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&full_a[s]), kBM);
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        mbar_init(smem_addr(&acc_full), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;

    auto fail = [&]() {
        s_abort = 1;
        atomicOr(a.err, 2);
    };

    if (warp == 0) {
        // ------------------------------------------------ x tiles (TMA)
        if (lane == 0) {
            for (int i = 0; i < nst; ++i) {
                const int s = i % kStages, u = i / kStages;
                if (u > 0 && !mbar_wait_bounded(smem_addr(&empty[s]), (u - 1) & 1, s_abort ? kDrain : kWait))
                    fail();
                const uint32_t bar = smem_addr(&full_b[s]);
                mbar_arrive_expect_tx(bar, kBSlot);
                tma_load_2d(b_ring + s * kBSlot, &xmap, i * kBK, m0, bar);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            for (int i = 0; i < nst; ++i) {
                const int s = i % kStages, u = i / kStages;
                if (!mbar_wait_bounded(smem_addr(&full_b[s]), u & 1, s_abort ? kDrain : kWait))
                    fail();
                if (!mbar_wait_bounded(smem_addr(&full_a[s]), u & 1, s_abort ? kDrain : kWait))
                    fail();
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint64_t ad = sdesc_k128(a_ring + s * kASlot);
                const uint64_t bd = sdesc_k128(b_ring + s * kBSlot);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) // +32 bytes of K per step
                    mma_bf16(tmem, ad + 2u * k, bd + 2u * k, kIdesc, (i | k) != 0);
                mma_commit(smem_addr(&empty[s]));
            }
            mma_commit(smem_addr(&acc_full));
        }
    } else {
        // ------------------------------------------------ A tiles (dequant)
        const int r = threadIdx.x - 64; // row of the tile, 0..127
        const int n = n0 + r;
        const bool valid = n < a.N;
        const uint32_t *qrow = a.qw + (size_t)(valid ? n : 0) * (a.K >> 3);
        const uint16_t *srow = a.sc + (size_t)(valid ? n : 0) * (a.K >> 5);
        const uint32_t rowoff = (uint32_t)r * 128u;
        const uint32_t sw = (uint32_t)(r & 7);
        uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
        uint32_t s01 = 0u;
        auto load = [&](int i) {
            if (valid) {
                w0 = ldg_stream_v4(qrow + 8 * i);
                w1 = ldg_stream_v4(qrow + 8 * i + 4);
                s01 = ldg_nc_u32(srow + 2 * i);
            }
        };
        load(0);
        for (int i = 0; i < nst; ++i) {
            const int s = i % kStages, u = i / kStages;
            const uint4 c0 = w0, c1 = w1;
            const uint32_t st = s01;
            if (i + 1 < nst)
                load(i + 1); // next stage's codes in flight while this one is stored
            if (u > 0 && !mbar_wait_bounded(smem_addr(&empty[s]), (u - 1) & 1, s_abort ? kDrain : kWait))
                fail();
            const uint32_t base = a_ring + s * kASlot + rowoff;
            const uint32_t sa = valid ? __byte_perm(st, st, 0x1010) : 0u; // group 2i, both halves
            const uint32_t sb = valid ? __byte_perm(st, st, 0x3232) : 0u; // group 2i + 1
            const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t p01, p23, p45, p67;
                dequant_word(words[j], j < 4 ? sa : sb, p01, p23, p45, p67);
                if (!valid)
                    p01 = p23 = p45 = p67 = 0u;
                sts128(base + ((((uint32_t)j) ^ sw) << 4), p01, p23, p45, p67);
            }
            // Generic-proxy stores must be visible to the tensor core (async proxy).
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(smem_addr(&full_a[s]));
        }

        // ------------------------------------------------ epilogue
        if (!mbar_wait_bounded(smem_addr(&acc_full), 0, s_abort ? kDrain : kWait))
            fail();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int q = warp & 3;               // TMEM lane quarter this warp may read
        const int row = n0 + 32 * q + lane;   // weight row = output column of y
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            uint32_t v[32];
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                         "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                         "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                         : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                           "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                           "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
                           "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                           "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]),
                           "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                         : "r"(taddr + (uint32_t)c0));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (row < a.N) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int m = m0 + c0 + j;
                    if (m < a.M)
                        a.y[(size_t)m * a.N + row] = __uint_as_float(v[j]);
                }
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

} // namespace

cudaError_t run_prefill(float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int M,
                        int N, int K, int num_sms, int *err, cudaStream_t s)
{
    (void)num_sms;
    if (K % kBK != 0 || N % 16 != 0)
        return cudaErrorNotSupported;
    auto enc = encoder();
    if (!enc)
        return cudaErrorNotSupported;
    CUtensorMap xmap;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBN};
    cuuint32_t es[2] = {1, 1};
    if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemm_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem);
    if (e != cudaSuccess)
        return e;
    PrefillArgs a;
    a.y = y;
    a.qw = qw;
    a.sc = sc;
    a.err = err;
    a.M = M;
    a.N = N;
    a.K = K;
    const dim3 grid((N + kBM - 1) / kBM, (M + kBN - 1) / kBN);
    gemm_prefill_kernel<<<grid, kThreads, kSmem, s>>>(a, xmap);
    return cudaGetLastError();
}

} // namespace w4
