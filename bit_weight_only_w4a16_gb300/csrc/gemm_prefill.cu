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
// y[m][n] = sum_k x[m][k] * bf16_rne((code(n,k) - 8) * step(n, k/group)), fp32
// accumulate. Rounding each weight to bf16 (relative error <= 2^-9) keeps the
// result within 2e-3 * sum|w x|.
//
// Persistent kernel, one CTA per SM. A work item is a tile of 128 weight rows
// (the MMA's M, TMEM lanes) x 256 tokens (the MMA's N) over a range of K. Whole
// tiles are dealt round-robin to the CTAs for as many full rounds as there are;
// the remaining tiles are split along K into S parts so that the last round
// spreads over all SMs (S = 1 when the tiles divide evenly). Every role walks
// the same item sequence.
//   warp 0     : TMA of the x tiles (256 tokens x 64 k, 128-byte swizzle) - B operand
//   warp 1     : allocates 512 TMEM columns (two accumulators); lane 0 issues
//                tcgen05.mma (4 x K=16 per stage) and commits each stage's slot
//                back to the producers and each finished accumulator to the epilogue
//   warps 2-9  : two threads per weight row (32 k each): codes and step six
//                stages ahead in registers, dequantized to bf16 into the K-major
//                128-byte-swizzle A tile the MMA reads
//   warps 10-13: epilogue: tcgen05.ld of their 32 TMEM lanes, coalesced fp32
//                stores of y, or for a split tile of its partial.
// A second kernel adds the S partials of each split tile in split order (a
// fixed order: the result does not depend on timing) and writes y.
// The epilogue of item j overlaps the MMAs of item j+1 (double-buffered TMEM).
// Every wait is bounded; a timeout sets the device error word and the kernel
// still drains its copies and MMAs and frees TMEM before returning.
#include "common.cuh"
#include "internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace w4 {

namespace {

constexpr int kBM = 128; // weight rows per tile
constexpr int kBN = 256; // tokens per tile
constexpr int kBK = 64;  // k per stage
constexpr int kStages = 4;
constexpr int kDqWarps = 8;
constexpr int kDqAhead = 6; // k-stages of codes in flight per dequant thread
constexpr int kEpiWarp0 = 2 + kDqWarps; // first epilogue warp
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kASlot = kBM * kBK * 2; // 16 KiB
constexpr int kBSlot = kBN * kBK * 2; // 32 KiB
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr size_t kSmem = (size_t)kStages * (kASlot + kBSlot) + 1024;
constexpr int kTileFloats = kBM * kBN;
constexpr int kWait = 1 << 16;
constexpr int kDrain = 64;

// tcgen05 instruction descriptor, kind::f16: fp32 D, bf16 A and B, both
// K-major, N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

// Shared-memory matrix descriptor: K-major operand in the 128-byte-swizzle
// layout (8-row x 128-byte atoms, 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;           // leading byte offset (unused for this layout): 16 B
    d |= (uint64_t)(1024 >> 4) << 32; // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;           // descriptor version
    d |= (uint64_t)2 << 61;           // 128-byte swizzle
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
    const uint32_t lo = w & 0x0F0F0F0Fu;             // codes k0 k2 k4 k6 in bytes 0..3
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;      // codes k1 k3 k5 k7
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
    float *ws; // split partials, one kTileFloats slot per (split tile, split)
    int *err;
    int M, N, K;
    int lg;       // one step per 32 << lg codes
    int tiles_n;  // 128-row weight tiles
    int tiles;    // tiles_n * 256-token tiles
    int full;     // tiles computed whole (the first full rounds)
    int S;        // K splits of each of the remaining tiles
    int items;    // full + (tiles - full) * S
};

// Item i -> tile t (weight tile t % tiles_n, token tile t / tiles_n), its split
// s of S (S = 1 for whole tiles). Consecutive items share the token tile, so
// CTAs working at the same time read the same x rows.
struct Item {
    int t, s, S;
};
__device__ __forceinline__ Item item_of(const PrefillArgs &a, int i)
{
    Item it;
    if (i < a.full) {
        it.t = i;
        it.s = 0;
        it.S = 1;
    } else {
        const int j = i - a.full, rem = a.tiles - a.full;
        it.t = a.full + j % rem;
        it.s = j / rem;
        it.S = a.S;
    }
    return it;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap xmap)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full_a[kStages], full_b[kStages], empty[kStages];
    __shared__ __align__(8) unsigned long long acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t a_ring = smem_addr(smem);
    const uint32_t b_ring = a_ring + kStages * kASlot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nst = a.K / kBK; // k-stages of a whole row

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&full_a[s]), kDqWarps); // one arrival per dequant warp
            mbar_init(smem_addr(&full_b[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&acc_full[b]), 1);
            mbar_init(smem_addr(&acc_empty[b]), 4); // one arrival per epilogue warp
        }
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
    // The split-K reduction kernel may start launching now; it waits for this
    // grid to complete before it reads the partials.
    pdl_launch_dependents();

    auto fail = [&]() {
        s_abort = 1;
        atomicOr(a.err, 2);
    };
    auto wait = [&](unsigned long long &bar, uint32_t parity) {
        if (!mbar_wait_bounded(smem_addr(&bar), parity, s_abort ? kDrain : kWait))
            fail();
    };
    auto k_begin = [&](const Item &it, int s) { return (int)((long long)nst * s / it.S); };

    if (warp == 0) {
        // ------------------------------------------------ x tiles (TMA)
        if (lane == 0) {
            uint32_t g = 0;
            for (int i = blockIdx.x; i < a.items; i += gridDim.x) {
                const Item it = item_of(a, i);
                const int k0 = k_begin(it, it.s), k1 = k_begin(it, it.s + 1);
                const int m0 = (it.t / a.tiles_n) * kBN;
                for (int st = k0; st < k1; ++st, ++g) {
                    const uint32_t slot = g % kStages, u = g / kStages;
                    if (u > 0)
                        wait(empty[slot], (u - 1) & 1);
                    const uint32_t bar = smem_addr(&full_b[slot]);
                    mbar_arrive_expect_tx(bar, kBSlot);
                    tma_load_2d(b_ring + slot * kBSlot, &xmap, st * kBK, m0, bar);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t g = 0, j = 0;
            for (int i = blockIdx.x; i < a.items; i += gridDim.x, ++j) {
                const Item it = item_of(a, i);
                const int k0 = k_begin(it, it.s), k1 = k_begin(it, it.s + 1);
                const uint32_t b = j & 1, uj = j >> 1;
                if (j >= 2)
                    wait(acc_empty[b], (uj - 1) & 1);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acc = tmem + b * kBN;
                for (int st = k0; st < k1; ++st, ++g) {
                    const uint32_t slot = g % kStages, u = g / kStages;
                    wait(full_b[slot], u & 1);
                    wait(full_a[slot], u & 1);
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint64_t ad = sdesc_k128(a_ring + slot * kASlot);
                    const uint64_t bd = sdesc_k128(b_ring + slot * kBSlot);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) // +32 bytes of K per step
                        mma_bf16(acc, ad + 2u * k, bd + 2u * k, kIdesc, (st > k0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_addr(&empty[slot]));
                }
                mma_commit(smem_addr(&acc_full[b]));
            }
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ A tiles (dequant)
        const int d = threadIdx.x - 64;
        const int r = d & (kBM - 1); // row of the tile
        const int h = d >> 7;        // which 32 k of the stage: group 2st + h
        const uint32_t rowoff = (uint32_t)r * 128u;
        const uint32_t sw = (uint32_t)(r & 7);
        uint32_t g = 0;
        for (int i = blockIdx.x; i < a.items; i += gridDim.x) {
            const Item it = item_of(a, i);
            const int k0 = k_begin(it, it.s), k1 = k_begin(it, it.s + 1);
            const int n = (it.t % a.tiles_n) * kBM + r;
            const bool valid = n < a.N;
            const uint32_t *qrow = a.qw + (size_t)(valid ? n : 0) * (a.K >> 3) + 4 * h;
            const uint16_t *srow = a.sc + (size_t)(valid ? n : 0) * (a.K >> (5 + a.lg));
            // Codes and step of the next kDqAhead stages in flight: stage st lives
            // in register set (st - k0) % kDqAhead, refilled with st + kDqAhead as
            // soon as it is consumed (no register copies, which would wait for the
            // load in flight).
            uint4 cw[kDqAhead];
            uint32_t cs[kDqAhead];
            auto load = [&](int st, uint4 &w, uint32_t &s1) {
                if (valid && st < k1) {
                    w = ldg_stream_v4(qrow + 8 * st);
                    s1 = ldg_nc_u16(srow + ((2 * st + h) >> a.lg));
                } else {
                    w = make_uint4(0u, 0u, 0u, 0u);
                    s1 = 0u;
                }
            };
#pragma unroll
            for (int u = 0; u < kDqAhead; ++u)
                load(k0 + u, cw[u], cs[u]);
            for (int base = k0; base < k1; base += kDqAhead) {
#pragma unroll
                for (int u = 0; u < kDqAhead; ++u) {
                    const int st = base + u;
                    if (st < k1) {
                        const uint32_t slot = g % kStages, uu = g / kStages;
                        if (uu > 0)
                            wait(empty[slot], (uu - 1) & 1);
                        const uint32_t dst = a_ring + slot * kASlot + rowoff;
                        const uint32_t step2 = valid ? (cs[u] | (cs[u] << 16)) : 0u;
                        const uint32_t words[4] = {cw[u].x, cw[u].y, cw[u].z, cw[u].w};
#pragma unroll
                        for (int jw = 0; jw < 4; ++jw) {
                            uint32_t p01, p23, p45, p67;
                            dequant_word(words[jw], step2, p01, p23, p45, p67);
                            if (!valid)
                                p01 = p23 = p45 = p67 = 0u;
                            sts128(dst + ((((uint32_t)(4 * h + jw)) ^ sw) << 4), p01, p23, p45, p67);
                        }
                        // Generic-proxy stores must be visible to the tensor core
                        // (async proxy); then one arrival for the warp.
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(smem_addr(&full_a[slot]));
                        load(st + kDqAhead, cw[u], cs[u]);
                        ++g;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3; // TMEM lane quarter this warp may read
        uint32_t j = 0;
        for (int i = blockIdx.x; i < a.items; i += gridDim.x, ++j) {
            const Item it = item_of(a, i);
            const uint32_t b = j & 1, uj = j >> 1;
            const int n0 = (it.t % a.tiles_n) * kBM, m0 = (it.t / a.tiles_n) * kBN;
            const bool split = it.S > 1;
            wait(acc_full[b], uj & 1);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int rl = 32 * q + lane; // row of the tile
            const int row = n0 + rl;      // weight row = output column of y
            // A split tile's partial goes to its slot, token-major [256][128].
            float *part = split ? a.ws + ((size_t)(it.t - a.full) * it.S + it.s) * kTileFloats : nullptr;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + b * kBN;
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
                if (split) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        part[(c0 + jj) * kBM + rl] = __uint_as_float(v[jj]);
                } else if (row < a.N) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int m = m0 + c0 + jj;
                        if (m < a.M)
                            a.y[(size_t)m * a.N + row] = __uint_as_float(v[jj]);
                    }
                }
            }
            // This accumulator may be overwritten by the MMAs of item j + 2.
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&acc_empty[b]));

        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// y of the split tiles: the S partials of each, added in split order. One CTA
// of 256 threads per (split tile, 32-token slice); thread i handles 4 weight
// rows (float4) of 4 tokens of the slice.
__global__ void __launch_bounds__(256)
prefill_split_reduce_kernel(float *__restrict__ y, const float *__restrict__ ws, int M, int N, int tiles_n,
                            int full, int S)
{
    pdl_wait(); // the partials are complete and visible
    const int st = blockIdx.x; // split tile index
    const int t = full + st;
    const int n0 = (t % tiles_n) * kBM, m0 = (t / tiles_n) * kBN;
    const int r4 = 4 * (threadIdx.x & 31);
    const int tok0 = blockIdx.y * 32 + (threadIdx.x >> 5) * 4;
    const float4 *base = reinterpret_cast<const float4 *>(ws + (size_t)st * S * kTileFloats);
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = __ldcs(base + ((size_t)s * kTileFloats + (size_t)(tok0 + u) * kBM + r4) / 4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc[u].x += v[u].x;
            acc[u].y += v[u].y;
            acc[u].z += v[u].z;
            acc[u].w += v[u].w;
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int m = m0 + tok0 + u;
        if (m >= M)
            continue;
        const float o[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (n0 + r4 + c < N)
                y[(size_t)m * N + n0 + r4 + c] = o[c];
    }
}

cudaError_t launch(const PrefillArgs &a, const uint16_t *x, int grid, cudaStream_t s)
{
    auto enc = tmap_encoder();
    if (!enc)
        return cudaErrorNotSupported;
    CUtensorMap xmap;
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
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
    gemm_prefill_kernel<<<grid, kThreads, kSmem, s>>>(a, xmap);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.full == a.tiles)
        return e;
    // Programmatic dependent launch: the reduction's CTAs are placed while the
    // GEMM's last tiles finish.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.tiles - a.full, kBN / 32);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_split_reduce_kernel, a.y, (const float *)a.ws, a.M, a.N, a.tiles_n,
                              a.full, a.S);
}

} // namespace

PrefillPlan plan_prefill(int M, int N, int K, int num_sms, size_t ws_floats)
{
    // Whole tiles for every full round of the SMs; the tiles of the last,
    // partial round are split along K into S parts (S = SMs / remaining tiles,
    // at most 4 and at most the number of k-stages) when the partials fit the
    // scratch.
    PrefillPlan p;
    const int nst = K / kBK;
    const int tiles = ((N + kBM - 1) / kBM) * ((M + kBN - 1) / kBN);
    p.full = tiles - tiles % num_sms;
    const int rem = tiles - p.full;
    p.S = 1;
    if (rem > 0) {
        int S = num_sms / rem;
        S = S < 4 ? S : 4;
        S = S < nst ? S : nst;
        while (S > 1 && (size_t)rem * S * kTileFloats > ws_floats)
            --S;
        if (S > 1)
            p.S = S;
        else
            p.full = tiles;
    }
    const int items = p.full + (tiles - p.full) * p.S;
    p.grid = items < num_sms ? items : num_sms;
    p.bn = kBN;
    p.ok = true;
    return p;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
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

cudaError_t run_prefill(const PrefillPlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                        const uint16_t *sc, int M, int N, int K, int lg, float *ws, int *err, cudaStream_t s)
{
    if (K % kBK != 0 || N % 16 != 0 || !p.ok)
        return cudaErrorNotSupported;
    PrefillArgs a;
    a.y = y;
    a.qw = qw;
    a.sc = sc;
    a.lg = lg;
    a.ws = ws;
    a.err = err;
    a.M = M;
    a.N = N;
    a.K = K;
    a.tiles_n = (N + kBM - 1) / kBM;
    a.tiles = a.tiles_n * ((M + kBN - 1) / kBN);
    a.full = p.full;
    a.S = p.S;
    a.items = p.full + (a.tiles - p.full) * p.S;
    return launch(a, x, p.grid, s);
}

} // namespace w4
