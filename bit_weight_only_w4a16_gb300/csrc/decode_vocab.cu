// Vocabulary-sized decode GEMV (M = 1, optional fused greedy pick) with the
// weights landed in shared memory by tensor copies.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
// (decode reads every weight once, straight from the packed 4-bit words, and
// multiplies in registers without a 16-bit copy) and Step 2 (the tied 4-bit
// embedding doubles as the output layer, read once per token with the greedy
// pick).
//
// GB300 design. A 262144 x 1536 projection streams 226 MB with no dependency
// chain inside, so what limits it is the bytes in flight per SM and the issue
// rate. The register-preload form holds its in-flight tiles in registers (4
// tiles a warp, 115 registers, 16 warps per SM: ~74 KB in flight). Here each
// warp owns two shared-memory slots, each one half of a 16-row block (6 tiles
// of 128 codes per row, 6 KB of codes), filled by ONE 3-D tensor copy issued by
// the warp's lane 0 and completing on the slot's mbarrier. While the warp
// computes one slot the other is in flight: 16 warps x 6 KB = 96 KB in flight
// per SM, no registers held for it, and each tile costs the same instructions
// as before with shared-memory loads (short, fixed latency) in place of
// global ones.
//
// Layout. The copy box is {32 words, 3 chunks, 16 rows} with the hardware's
// 128-byte swizzle: 16-byte granule q of 128-byte line L (L = 3 * row + chunk)
// lands at granule q ^ (L & 7). A warp's 128-bit code load for one row is read
// by 8 lanes at a time (rows of mma lanes g = 2p and 2p + 1, t = 0..3); mma row
// g holds weight row perm(g) = (g >> 1) + 4 * (g & 1) (and + 8 for rows
// g + 8), so the two rows of a phase are 4 apart, their lines 12 apart, and bit
// 2 of L & 7 differs: the 8 lanes touch 8 different granules, all 32 banks
// once.
//
// Inner product as in the other decode kernels: exact (code - 8) bf16 x bf16
// m16n8k16 mma with fp32 accumulate; lane (g, t) holds group 4 * tile + t of
// its two rows; B column s carries x restricted to group slot s; steps are
// applied per (row, group) in fp32 (they come from global memory, one slot
// ahead, since a steps row is not a multiple of 16 bytes for every group size).
#include "common.cuh"
#include "internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

namespace w4 {

namespace {

constexpr int kTs = 6;                // tiles per slot (half a row block at K = 1536)
constexpr int kLines = kTs / 2;       // 128-byte lines per row and slot
constexpr int kSlotBytes = 16 * kTs * 64;
constexpr int kStepBytes = 16 * kTs * 4 * 2; // group 32: 4 bf16 steps per tile and row
constexpr int kWarps = 16;
constexpr int kSlots = 2;             // per warp
constexpr int kWaitLimit = 1 << 16;   // tests (each up to ~20 us) before a wait gives up
constexpr int kDrainLimit = 64;       // tests per in-flight copy once a wait has given up

struct VocabArgs {
    float *y;
    const uint16_t *x;
    const uint16_t *sc;
    unsigned long long *keys; // per-CTA argmax keys or null
    int *err;                 // device error word: bit 0 set when a slot wait ran out
    const int32_t *forced;    // forced next token (>= 0: no weight is read) or null
    int N, K, lg;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
                 "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar,
                                            uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
                 "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ int perm_row(int g) { return (g >> 1) + 4 * (g & 1); }

// Shared-memory byte offset of the 16 bytes of tile l (0..kTs-1), group slot t,
// weight row r of a slot (swizzled as the copy lands it).
__device__ __forceinline__ uint32_t code_off(int r, int l, int t)
{
    const int L = r * kLines + (l >> 1);
    const int q = 4 * (l & 1) + t;
    return (uint32_t)(L * 128 + ((q ^ (L & 7)) << 4));
}

// G32: the slot's steps arrive by a second tensor copy ({24 steps, 16 rows},
// one 48-byte run per row) and are read from shared memory; other group sizes
// (a steps row of K/group bf16 is not always a multiple of 16 bytes, which a
// tensor copy needs) load theirs from global memory one slot ahead.
template <bool ARGMAX, bool G32>
__global__ void __launch_bounds__(kWarps * 32, 1)
w4_decode_vocab_kernel(const VocabArgs a, const __grid_constant__ CUtensorMap codes,
                       const __grid_constant__ CUtensorMap steps)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long bars[kWarps * kSlots];
    __shared__ unsigned long long ck;
    __shared__ int s_abort;
    // Slots on a 1024-byte boundary (the swizzle pattern's period).
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    if (ARGMAX && a.forced != nullptr && *a.forced >= 0) {
        // The next token is forced: no weight is read, y is left as it was, and
        // the pick kernel writes the forced token (after this grid completes).
        pdl_launch_dependents();
        pdl_wait();
        return;
    }

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nrb = a.N >> 4;
    const int T = a.K >> 7, halves = T / kTs;
    const int GW = gridDim.x * kWarps, gw = blockIdx.x * kWarps + warp;
    const int nmine = nrb > gw ? (nrb - gw + GW - 1) / GW : 0;
    const int nslots = nmine * halves; // slot fills of this warp, in order

    uint8_t *wslots = smem + (size_t)warp * kSlots * kSlotBytes;
    const uint32_t wslot0 = smem_addr(wslots);
    unsigned char *ssteps = smem + (size_t)kWarps * kSlots * kSlotBytes; // G32 steps slots
    const uint32_t wstep0 = smem_addr(ssteps + (size_t)warp * kSlots * kStepBytes);
    uint4 *xs = reinterpret_cast<uint4 *>(ssteps + (G32 ? (size_t)kWarps * kSlots * kStepBytes : 0));
    const int nchunk = a.K >> 3;
    uint4 *zs = xs + nchunk + 2;

    const uint32_t bar0 = smem_addr(&bars[warp * kSlots]);
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        for (int i = 0; i < kSlots; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        s_abort = 0;
        ck = 0ull;
    }
    __syncwarp();

    // Slot fill f (f = 0, 1, ...) of this warp: row block gw + (f / halves) * GW,
    // half f % halves, into slot f % kSlots.
    auto fill = [&](int f) {
        const int rb = gw + (f / halves) * GW, h = f % halves;
        const uint32_t bar = bar0 + 8u * (f % kSlots);
        mbar_arrive_expect_tx(bar, (uint32_t)(kSlotBytes + (G32 ? kStepBytes : 0)));
        tma_load_3d(wslot0 + (uint32_t)((f % kSlots) * kSlotBytes), &codes, 0, h * kLines, rb * 16, bar, policy);
        if (G32)
            tma_load_2d(wstep0 + (uint32_t)((f % kSlots) * kStepBytes), &steps, h * kTs * 4, rb * 16, bar, policy);
    };
    if (lane == 0)
        for (int f = 0; f < kSlots && f < nslots; ++f)
            fill(f);
    if (threadIdx.x == 32)
        prefetch_l2_bulk(a.x, (uint32_t)(a.K * 2));
    pdl_launch_dependents();
    pdl_wait();

    // x, permuted into the B-operand pair order; a zero region for the lanes
    // that feed zero columns (granules on other banks than x's). When every x
    // value is exact in fp16 the CTA runs the fp16 unpack (fewer ALU
    // instructions per code; the same products and fp32 sums), else the bf16 one.
    bool exact = true;
    for (int i = threadIdx.x; i < nchunk; i += blockDim.x) {
        const uint4 v = *reinterpret_cast<const uint4 *>(a.x + 8 * i);
        bf16x2_to_f16x2_exact(v.x, exact);
        bf16x2_to_f16x2_exact(v.y, exact);
        bf16x2_to_f16x2_exact(v.z, exact);
        bf16x2_to_f16x2_exact(v.w, exact);
    }
    const bool f16 = __syncthreads_and(exact) != 0;
    for (int i = threadIdx.x; i < nchunk; i += blockDim.x) {
        uint4 v = *reinterpret_cast<const uint4 *>(a.x + 8 * i);
        if (f16) {
            bool dummy = true;
            v = make_uint4(bf16x2_to_f16x2_exact(v.x, dummy), bf16x2_to_f16x2_exact(v.y, dummy),
                           bf16x2_to_f16x2_exact(v.z, dummy), bf16x2_to_f16x2_exact(v.w, dummy));
        }
        xs[i] = permute_x8(v);
    }
    if (threadIdx.x < 4)
        zs[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    const bool bsel = g < 4 && t == g;
    const uint4 *xlane = bsel ? xs + 4 * t : zs;
    const int xstep = bsel ? 16 : 0;

    // This lane's weight rows in a row block and their step pointers.
    const int rA = perm_row(g), rB = rA + 8;
    const int sstride = (a.K >> 5) >> a.lg;
    const int jt = 2 * (t & 1);
    uint32_t sa[2][kTs], sb[2][kTs];
    auto load_steps = [&](int f, auto bufc) {
        constexpr int buf = decltype(bufc)::value;
        if (G32)
            return; // landed with the codes
        const int rb = gw + (f / halves) * GW, h = f % halves;
        const uint16_t *pa = a.sc + (size_t)(rb * 16 + rA) * sstride;
        const uint16_t *pb = a.sc + (size_t)(rb * 16 + rB) * sstride;
#pragma unroll
        for (int l = 0; l < kTs; ++l) {
            const int j = 4 * (h * kTs + l) + jt; // first 32-code group of the lane's pair
            if (G32) {
                sa[buf][l] = ldg_nc_u32(pa + j);
                sb[buf][l] = ldg_nc_u32(pb + j);
            } else {
                sa[buf][l] = ldg_nc_u16(pa + (j >> a.lg));
                sb[buf][l] = ldg_nc_u16(pb + (j >> a.lg));
            }
        }
    };
    if (nslots > 0)
        load_steps(0, std::integral_constant<int, 0>{});

    float accA = 0.f, accB = 0.f;
    bool ok = true;         // warp-uniform: every slot wait so far completed
    int issued = nslots < kSlots ? nslots : kSlots, failed = -1;
    // One slot fill; BUF (compile-time) selects the step registers, so the two
    // sets stay in registers (fills alternate between them).
    auto consume = [&](auto bufc, auto f16c, int f) {
        constexpr int buf = decltype(bufc)::value;
        constexpr bool F16 = decltype(f16c)::value;
        const uint32_t stA = wstep0 + (uint32_t)((f % kSlots) * kStepBytes + rA * kTs * 8 + 2 * jt);
        const uint32_t stB = stA + 8u * 8u * kTs; // 8 rows on
        if (f + 1 < nslots)
            load_steps(f + 1, std::integral_constant<int, buf ^ 1>{});
        const uint32_t bar = bar0 + 8u * (f % kSlots);
        const uint32_t parity = (uint32_t)((f / kSlots) & 1);
        if (ok) {
            const bool done = mbar_wait_bounded(bar, parity, kWaitLimit);
            ok = __all_sync(0xFFFFFFFFu, done);
            if (!ok) {
                failed = f;
                if (lane == 0) {
                    atomicOr(a.err, 1);
                    s_abort = 1;
                }
            }
        }
        const uint32_t sbase = wslot0 + (uint32_t)((f % kSlots) * kSlotBytes);
        const int h = f % halves;
        const uint4 *xh = xlane + (size_t)xstep * h * kTs;
#pragma unroll
        for (int l = 0; l < kTs; l += 2) {
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, d0[4] = {0.f, 0.f, 0.f, 0.f};
            float c1[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 wa0 = lds128(sbase + code_off(rA, l, t)), wb0 = lds128(sbase + code_off(rB, l, t));
            const uint4 wa1 = lds128(sbase + code_off(rA, l + 1, t)), wb1 = lds128(sbase + code_off(rB, l + 1, t));
            const uint4 *xb = xh + xstep * l;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 b0 = xb[i], b1 = xb[xstep + i];
                if (F16) {
                    unpack_mma2_f16(c0, d0, (&wa0.x)[i], (&wb0.x)[i], b0.x, b0.y, b0.z, b0.w);
                    unpack_mma2_f16(c1, d1, (&wa1.x)[i], (&wb1.x)[i], b1.x, b1.y, b1.z, b1.w);
                } else {
                    unpack_mma2(c0, d0, (&wa0.x)[i], (&wb0.x)[i], b0.x, b0.y, b0.z, b0.w);
                    unpack_mma2(c1, d1, (&wa1.x)[i], (&wb1.x)[i], b1.x, b1.y, b1.z, b1.w);
                }
            }
            if (G32) {
                const uint32_t s0 = lds32(stA + 8u * l), s1 = lds32(stA + 8u * (l + 1));
                const uint32_t t0 = lds32(stB + 8u * l), t1 = lds32(stB + 8u * (l + 1));
                accA = fmaf(bf16lo_to_f32(s0), c0[0] + d0[0], accA);
                accA = fmaf(bf16hi_to_f32(s0), c0[1] + d0[1], accA);
                accB = fmaf(bf16lo_to_f32(t0), c0[2] + d0[2], accB);
                accB = fmaf(bf16hi_to_f32(t0), c0[3] + d0[3], accB);
                accA = fmaf(bf16lo_to_f32(s1), c1[0] + d1[0], accA);
                accA = fmaf(bf16hi_to_f32(s1), c1[1] + d1[1], accA);
                accB = fmaf(bf16lo_to_f32(t1), c1[2] + d1[2], accB);
                accB = fmaf(bf16hi_to_f32(t1), c1[3] + d1[3], accB);
            } else { // one step for both groups of the pair
                accA = fmaf(bf16lo_to_f32(sa[buf][l]), (c0[0] + d0[0]) + (c0[1] + d0[1]), accA);
                accB = fmaf(bf16lo_to_f32(sb[buf][l]), (c0[2] + d0[2]) + (c0[3] + d0[3]), accB);
                accA = fmaf(bf16lo_to_f32(sa[buf][l + 1]), (c1[0] + d1[0]) + (c1[1] + d1[1]), accA);
                accB = fmaf(bf16lo_to_f32(sb[buf][l + 1]), (c1[2] + d1[2]) + (c1[3] + d1[3]), accB);
            }
        }
        // Every lane's reads of this slot are done (their values are in
        // registers); lane 0 refills it with the warp's fill f + kSlots.
        __syncwarp();
        if (ok && f + kSlots < nslots) {
            if (lane == 0)
                fill(f + kSlots);
            ++issued;
        }
        if (h == halves - 1) { // row block done: lanes t, t ^ 1 hold slots (0,1), (2,3)
            const float vA = accA + __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
            const float vB = accB + __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
            const int rb = gw + (f / halves) * GW;
            if (t == 0) {
                const int rowA = rb * 16 + rA, rowB = rb * 16 + rB;
                a.y[rowA] = vA;
                a.y[rowB] = vB;
                if (ARGMAX) {
                    atomicMax(&ck, argmax_key(vA, (uint32_t)rowA));
                    atomicMax(&ck, argmax_key(vB, (uint32_t)rowB));
                }
            }
            accA = accB = 0.f;
        }
    };
    auto run = [&](auto f16c) {
        for (int f = 0; f < nslots; f += 2) {
            consume(std::integral_constant<int, 0>{}, f16c, f);
            if (f + 1 < nslots)
                consume(std::integral_constant<int, 1>{}, f16c, f + 1);
        }
    };
    if (f16)
        run(std::true_type{});
    else
        run(std::false_type{});

    // After a wait gave up: wait (bounded again) for this warp's copies still in
    // flight, so none lands in shared memory after the CTA has exited.
    if (failed >= 0 && lane == 0)
        for (int f = failed; f < issued; ++f)
            mbar_wait_bounded(bar0 + 8u * (f % kSlots), (uint32_t)((f / kSlots) & 1), kDrainLimit);

    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x == 0)
            a.keys[blockIdx.x] = ck;
    }
}

constexpr size_t kSmem = (size_t)kWarps * kSlots * kSlotBytes; // + steps (group 32), x, zero region, slack

// The decode sweep's long M = 1 projections (gate|up, down) with the same
// shared-memory slots: a CTA owns R consecutive 16-row blocks and all S = T/6
// six-tile slices of them ("units", R * S of them); warp w of W (16, or 8 when
// 16 warps' slots and x do not fit) takes units w, w + W, ... into its two
// slots. The slots' copies are issued when the CTA starts, before the wait on
// the previous call, so a CTA whose units fit its 2 W slots has its whole
// weight slice requested at once. After the wait x is
// staged, each warp computes its units from shared memory and leaves each
// unit's 16 row partials in shared memory; the partials of a row are added in
// slice order (deterministic). Group 32 only (steps by tensor copy).
// PL = 8 or 16 (Hadamard-rotated weights, blocks of 32 PL): the CTA forms the
// (hi, lo) rows of x H while staging x (norm = 1/sqrt(block)); B column s
// carries hi restricted to group slot s and column 4 + s the lo row, so lanes
// t and t + 2 hold the two rows' partials of the same groups, added with the
// slot pair.
template <int PL>
__global__ void __launch_bounds__(kWarps * 32, 1)
w4_decode_slab_kernel(const VocabArgs a, int R, float norm, const __grid_constant__ CUtensorMap codes,
                      const __grid_constant__ CUtensorMap steps)
{
    constexpr bool ROT = PL > 0;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long bars[kWarps * kSlots];
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5; // 16 warps, or 8 when 16 warps' slots and x do not fit
    const int g = lane >> 2, t = lane & 3;
    const int nrb = a.N >> 4;
    const int S = (a.K >> 7) / kTs;                 // six-tile slices per row
    const int rb0 = blockIdx.x * R;
    const int Rn = min(R, nrb - rb0);
    const int nunits = Rn * S;
    const int nmine = warp < nunits ? (nunits - warp + W - 1) / W : 0;

    const uint32_t wslot0 = smem_addr(smem + (size_t)warp * kSlots * kSlotBytes);
    unsigned char *ssteps = smem + (size_t)W * kSlots * kSlotBytes;
    const uint32_t wstep0 = smem_addr(ssteps + (size_t)warp * kSlots * kStepBytes);
    uint4 *xs = reinterpret_cast<uint4 *>(ssteps + (size_t)W * kSlots * kStepBytes); // [ROT ? 2 : 1][nchunk]
    const int nchunk = a.K >> 3;
    uint4 *zs = xs + (ROT ? 2 : 1) * nchunk + 2;
    float *red = reinterpret_cast<float *>(zs + 6); // [nunits][16]

    const uint32_t bar0 = smem_addr(&bars[warp * kSlots]);
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        for (int i = 0; i < kSlots; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // Fill f of this warp: unit warp + f * W = (row block r, slice h).
    auto fill = [&](int f) {
        const int u = warp + f * W, r = u / S, h = u - r * S;
        const uint32_t bar = bar0 + 8u * (f % kSlots);
        mbar_arrive_expect_tx(bar, (uint32_t)(kSlotBytes + kStepBytes));
        tma_load_3d(wslot0 + (uint32_t)((f % kSlots) * kSlotBytes), &codes, 0, h * kLines, (rb0 + r) * 16, bar,
                    policy);
        tma_load_2d(wstep0 + (uint32_t)((f % kSlots) * kStepBytes), &steps, h * kTs * 4, (rb0 + r) * 16, bar,
                    policy);
    };
    if (lane == 0)
        for (int f = 0; f < kSlots && f < nmine; ++f)
            fill(f);
    if (threadIdx.x == 32)
        prefetch_l2_bulk(a.x, (uint32_t)(a.K * 2));
    pdl_launch_dependents();
    pdl_wait();

    if (ROT) {
        stage_x_hadamard<(ROT ? PL : 8)>(xs, a.x, a.K, nchunk, norm);
    } else {
        // Up to kXL chunks of a thread in flight at once (6 a thread at
        // K = 12288 with 8 warps): one memory round trip, not one per chunk.
        constexpr int kXL = 6;
        for (int i0 = threadIdx.x; i0 < nchunk; i0 += kXL * blockDim.x) {
            uint4 v[kXL];
#pragma unroll
            for (int q = 0; q < kXL; ++q) {
                const int i = i0 + q * blockDim.x;
                v[q] = i < nchunk ? ldg_stream_v4(a.x + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < kXL; ++q) {
                const int i = i0 + q * blockDim.x;
                if (i < nchunk)
                    xs[i] = permute_x8(v[q]);
            }
        }
    }
    if (threadIdx.x < 4)
        zs[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // Lane (g, t) feeds B column g: x (the hi row) restricted to group slot t
    // when g == t, the lo row when g == t + 4 (rotated), else the zero region.
    const bool bsel = g < 4 && t == g;
    const bool blo = ROT && g >= 4 && t == g - 4;
    const uint4 *xlane = bsel ? xs + 4 * t : (blo ? xs + nchunk + 4 * t : zs);
    const int xstep = (bsel || blo) ? 16 : 0;
    const int rA = perm_row(g), rB = rA + 8;
    const int jt = 2 * (t & 1);

    bool ok = true;
    int issued = nmine < kSlots ? nmine : kSlots, failed = -1;
    for (int f = 0; f < nmine; ++f) {
        const uint32_t bar = bar0 + 8u * (f % kSlots);
        const uint32_t parity = (uint32_t)((f / kSlots) & 1);
        if (ok) {
            const bool done = mbar_wait_bounded(bar, parity, kWaitLimit);
            ok = __all_sync(0xFFFFFFFFu, done);
            if (!ok) {
                failed = f;
                if (lane == 0)
                    atomicOr(a.err, 1);
            }
        }
        const int u = warp + f * W, h = u % S;
        const uint32_t sbase = wslot0 + (uint32_t)((f % kSlots) * kSlotBytes);
        const uint32_t stA = wstep0 + (uint32_t)((f % kSlots) * kStepBytes + rA * kTs * 8 + 2 * jt);
        const uint32_t stB = stA + 8u * 8u * kTs;
        const uint4 *xh = xlane + (size_t)xstep * h * kTs;
        float accA = 0.f, accB = 0.f;
#pragma unroll
        for (int l = 0; l < kTs; l += 2) {
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, d0[4] = {0.f, 0.f, 0.f, 0.f};
            float c1[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 wa0 = lds128(sbase + code_off(rA, l, t)), wb0 = lds128(sbase + code_off(rB, l, t));
            const uint4 wa1 = lds128(sbase + code_off(rA, l + 1, t)), wb1 = lds128(sbase + code_off(rB, l + 1, t));
            const uint4 *xb = xh + xstep * l;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 b0 = xb[i], b1 = xb[xstep + i];
                unpack_mma2(c0, d0, (&wa0.x)[i], (&wb0.x)[i], b0.x, b0.y, b0.z, b0.w);
                unpack_mma2(c1, d1, (&wa1.x)[i], (&wb1.x)[i], b1.x, b1.y, b1.z, b1.w);
            }
            const uint32_t s0 = lds32(stA + 8u * l), s1 = lds32(stA + 8u * (l + 1));
            const uint32_t t0 = lds32(stB + 8u * l), t1 = lds32(stB + 8u * (l + 1));
            accA = fmaf(bf16lo_to_f32(s0), c0[0] + d0[0], accA);
            accA = fmaf(bf16hi_to_f32(s0), c0[1] + d0[1], accA);
            accB = fmaf(bf16lo_to_f32(t0), c0[2] + d0[2], accB);
            accB = fmaf(bf16hi_to_f32(t0), c0[3] + d0[3], accB);
            accA = fmaf(bf16lo_to_f32(s1), c1[0] + d1[0], accA);
            accA = fmaf(bf16hi_to_f32(s1), c1[1] + d1[1], accA);
            accB = fmaf(bf16lo_to_f32(t1), c1[2] + d1[2], accB);
            accB = fmaf(bf16hi_to_f32(t1), c1[3] + d1[3], accB);
        }
        __syncwarp();
        if (ok && f + kSlots < nmine) {
            if (lane == 0)
                fill(f + kSlots);
            ++issued;
        }
        // Lanes t, t ^ 1 hold group slots (0, 1) and (2, 3) of the unit's rows
        // (rotated: lanes t + 2 the lo row's).
        float vA = accA + __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
        float vB = accB + __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
        if (ROT) {
            vA += __shfl_xor_sync(0xFFFFFFFFu, vA, 2);
            vB += __shfl_xor_sync(0xFFFFFFFFu, vB, 2);
        }
        if (t == 0) {
            red[u * 16 + rA] = vA;
            red[u * 16 + rB] = vB;
        }
    }
    if (failed >= 0 && lane == 0)
        for (int f = failed; f < issued; ++f)
            mbar_wait_bounded(bar0 + 8u * (f % kSlots), (uint32_t)((f / kSlots) & 1), kDrainLimit);
    __syncthreads();

    // Each row's slices, added in slice order.
    float *yb = a.y + (size_t)rb0 * 16;
    for (int o = threadIdx.x; o < Rn * 16; o += blockDim.x) {
        const float *p = red + (o >> 4) * S * 16 + (o & 15);
        float v = p[0];
        for (int h = 1; h < S; ++h)
            v += p[16 * h];
        yb[o] = v;
    }
}


// ------------------------------------------------------------ M <= 8 ----
//
// The same shared-memory slots for 2..8 x-rows. The mma's eight B columns are
// the x rows (rows M..7 read a zero region), so each mma must stay inside one
// 32-code group: lane (g, t) reads word t of a group for its two weight rows
// with 32-bit shared loads straight out of the swizzled slot (the 8 rows of a
// load land on 8 different 16-byte granules, so the 32 lanes touch 32 banks),
// and the two mmas of the group chain into one accumulator that is scaled by
// the group's steps in fp32. Per 16 x 128 tile this is the M = 1 form's
// unpack and mma count with 8 code loads in place of 2 and 16 step FMAs.
// x rows are staged in shared memory permuted into the pair order, chunk c of
// row m at c ^ (4 (m & 1)) so that the 8 lanes of a 128-bit load phase (rows
// g, g + 1) hit different banks.
// Vocabulary sizes: one CTA per SM, warp gw of the grid walks row blocks gw,
// gw + GW, ..., each as S consecutive six-tile units through its two slots,
// and stores a row block's outputs (and argmax keys) after its last unit.
// (Measured on GB300: 262144 x 1536 with the pick 89.6 -> 53.8 us at M = 8,
// 87.6 -> 52.4 us at M = 4, 56.0 -> 46.9 us at M = 2 against the register
// forms. The same form with a CTA owning a few row blocks was slower than the
// register forms on every decode-sweep shape at M = 8: a warp's six-tile unit
// is too long a serial chain at M = 8 when a CTA holds only a few units.)
struct Slots8Args {
    float *y;
    const uint16_t *x;
    unsigned long long *keys; // per-(x-row, CTA) argmax keys or null
    int *err;                 // device error word: bit 0 set when a slot wait ran out
    int M, N, K;
};

template <bool ARGMAX>
__global__ void __launch_bounds__(kWarps * 32, 1)
w4_decode_slots8_kernel(const Slots8Args a, const __grid_constant__ CUtensorMap codes,
                        const __grid_constant__ CUtensorMap steps)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long bars[kWarps * kSlots];
    __shared__ unsigned long long ck[8];
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nrb = a.N >> 4;
    const int S = (a.K >> 7) / kTs; // six-tile units per row
    const int GW = gridDim.x * W, gw = blockIdx.x * W + warp;
    const int nmine = (nrb > gw ? (nrb - gw + GW - 1) / GW : 0) * S;
    // Unit f of this warp: row block rb, unit h of the row.
    auto unit_of = [&](int f, int &rb, int &h) {
        rb = gw + (f / S) * GW;
        h = f % S;
    };

    const uint32_t wslot0 = smem_addr(smem + (size_t)warp * kSlots * kSlotBytes);
    unsigned char *ssteps = smem + (size_t)W * kSlots * kSlotBytes;
    const uint32_t wstep0 = smem_addr(ssteps + (size_t)warp * kSlots * kStepBytes);
    const int cpr = a.K >> 3, nx = a.M * cpr;
    uint4 *xs = reinterpret_cast<uint4 *>(ssteps + (size_t)W * kSlots * kStepBytes); // [M][cpr]
    uint4 *zs = xs + nx;                                                               // 16 zero chunks

    const uint32_t bar0 = smem_addr(&bars[warp * kSlots]);
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        for (int i = 0; i < kSlots; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_mbar_init();
    }
    if (ARGMAX && threadIdx.x < 8)
        ck[threadIdx.x] = 0ull;
    __syncwarp();
    auto fill = [&](int f) {
        int rb, h;
        unit_of(f, rb, h);
        const uint32_t bar = bar0 + 8u * (f % kSlots);
        mbar_arrive_expect_tx(bar, (uint32_t)(kSlotBytes + kStepBytes));
        tma_load_3d(wslot0 + (uint32_t)((f % kSlots) * kSlotBytes), &codes, 0, h * kLines, rb * 16, bar, policy);
        tma_load_2d(wstep0 + (uint32_t)((f % kSlots) * kStepBytes), &steps, h * kTs * 4, rb * 16, bar, policy);
    };
    if (lane == 0)
        for (int f = 0; f < kSlots && f < nmine; ++f)
            fill(f);
    if (threadIdx.x == 32)
        prefetch_l2_bulk(a.x, (uint32_t)(nx * 16));
    pdl_launch_dependents();
    pdl_wait();

    // x rows, permuted and bank-swizzled. When every value is exact in fp16
    // and a thread holds at most 4 chunks (kept in registers between the check
    // and the store), the CTA stages fp16 and runs the fp16 unpack.
    const bool few = nx <= 4 * (int)blockDim.x;
    bool exact = few;
    uint4 v[4];
    if (few) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            if (i < nx) {
                v[q] = permute_x8(*reinterpret_cast<const uint4 *>(a.x + 8 * i));
                bf16x2_to_f16x2_exact(v[q].x, exact);
                bf16x2_to_f16x2_exact(v[q].y, exact);
                bf16x2_to_f16x2_exact(v[q].z, exact);
                bf16x2_to_f16x2_exact(v[q].w, exact);
            }
        }
    }
    const bool f16 = __syncthreads_and(exact) != 0;
    if (few) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = threadIdx.x + q * blockDim.x;
            if (i < nx) {
                const int m = i / cpr, c = i - m * cpr;
                uint4 o = v[q];
                if (f16) {
                    bool d = true;
                    o = make_uint4(bf16x2_to_f16x2_exact(o.x, d), bf16x2_to_f16x2_exact(o.y, d),
                                   bf16x2_to_f16x2_exact(o.z, d), bf16x2_to_f16x2_exact(o.w, d));
                }
                xs[m * cpr + (c ^ (4 * (m & 1)))] = o;
            }
        }
    } else {
        // Many chunks a thread: all of them in flight at once as asynchronous
        // 16-byte copies into their swizzled places, then each thread permutes
        // its own chunks in place (bf16).
        const uint32_t base = smem_addr(xs);
        int m = 0, c = threadIdx.x;
        while (c >= cpr) {
            c -= cpr;
            ++m;
        }
        const int m_first = m, c_first = c;
        for (int i = threadIdx.x; i < nx; i += blockDim.x) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                             base + 16u * (uint32_t)(m * cpr + (c ^ (4 * (m & 1))))),
                         "l"(a.x + 8 * (size_t)i)
                         : "memory");
            c += blockDim.x;
            while (c >= cpr) {
                c -= cpr;
                ++m;
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        m = m_first;
        c = c_first;
        for (int i = threadIdx.x; i < nx; i += blockDim.x) {
            uint4 *q = xs + m * cpr + (c ^ (4 * (m & 1)));
            *q = permute_x8(*q);
            c += blockDim.x;
            while (c >= cpr) {
                c -= cpr;
                ++m;
            }
        }
    }
    if (threadIdx.x < 16)
        zs[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // Lane constants. Weight rows rA, rB = rA + 8 of a row block (mma rows g,
    // g + 8); x row g (B column g) or the zero region; chunk offsets of group
    // slot j in a tile; per 128-byte line of row rA its offset and swizzle (row
    // rB is 24 lines on, with the same swizzle phase).
    const int rA = perm_row(g);
    const bool xreal = g < a.M;
    const uint4 *xb = xreal ? xs + g * cpr : zs;
    const int xst = xreal ? 16 : 0;
    const int sw = xreal ? 4 * (g & 1) : 0;
    int xo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        xo[j] = (4 * j + t) ^ sw;
    uint32_t coff[kLines], cx[kLines];
#pragma unroll
    for (int ll = 0; ll < kLines; ++ll) {
        const int L = rA * kLines + ll;
        coff[ll] = (uint32_t)(L * 128 + 4 * t);
        cx[ll] = (uint32_t)((L & 7) << 4);
    }
    const uint32_t stA = (uint32_t)(rA * kTs * 8), stB = stA + 8u * kTs * 8u;

    bool ok = true;
    int issued = nmine < kSlots ? nmine : kSlots, failed = -1;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    auto run = [&](auto f16c) {
        constexpr bool F16 = decltype(f16c)::value;
        for (int f = 0; f < nmine; ++f) {
            const uint32_t bar = bar0 + 8u * (f % kSlots);
            const uint32_t parity = (uint32_t)((f / kSlots) & 1);
            if (ok) {
                const bool done = mbar_wait_bounded(bar, parity, kWaitLimit);
                ok = __all_sync(0xFFFFFFFFu, done);
                if (!ok) {
                    failed = f;
                    if (lane == 0)
                        atomicOr(a.err, 1);
                }
            }
            int rb, h;
            unit_of(f, rb, h);
            const uint32_t sbase = wslot0 + (uint32_t)((f % kSlots) * kSlotBytes);
            const uint32_t stbase = wstep0 + (uint32_t)((f % kSlots) * kStepBytes);
            const uint4 *xh = xb + xst * h * kTs;
#pragma unroll
            for (int l = 0; l < kTs; ++l) {
                const uint2 sa = lds64(stbase + stA + 8u * l), sb = lds64(stbase + stB + 8u * l);
                const uint32_t cb = sbase + coff[l >> 1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t ad = cb + (((uint32_t)((4 * (l & 1) + j) << 4)) ^ cx[l >> 1]);
                    const uint32_t wa = lds32(ad), wb = lds32(ad + 24u * 128u);
                    const uint4 xv = xh[xst * l + xo[j]];
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    if (F16)
                        unpack_mma2_1_f16(c, wa, wb, xv.x, xv.y, xv.z, xv.w);
                    else
                        unpack_mma2_1(c, wa, wb, xv.x, xv.y, xv.z, xv.w);
                    const uint32_t pa = (j >> 1) ? sa.y : sa.x, pb = (j >> 1) ? sb.y : sb.x;
                    const float s_a = (j & 1) ? bf16hi_to_f32(pa) : bf16lo_to_f32(pa);
                    const float s_b = (j & 1) ? bf16hi_to_f32(pb) : bf16lo_to_f32(pb);
                    a0 = fmaf(s_a, c[0], a0);
                    a1 = fmaf(s_a, c[1], a1);
                    b0 = fmaf(s_b, c[2], b0);
                    b1 = fmaf(s_b, c[3], b1);
                }
            }
            // Every lane's reads of this slot are done; lane 0 refills it.
            __syncwarp();
            if (ok && f + kSlots < nmine) {
                if (lane == 0)
                    fill(f + kSlots);
                ++issued;
            }
            // Lane (g, t) holds x rows 2t, 2t + 1 of weight rows rA, rB.
            const int m0 = 2 * t, m1 = 2 * t + 1;
            if (h == S - 1) {
                const int rowA = rb * 16 + rA, rowB = rowA + 8;
                if (m0 < a.M) {
                    a.y[(size_t)m0 * a.N + rowA] = a0;
                    a.y[(size_t)m0 * a.N + rowB] = b0;
                    if (ARGMAX) {
                        atomicMax(&ck[m0], argmax_key(a0, (uint32_t)rowA));
                        atomicMax(&ck[m0], argmax_key(b0, (uint32_t)rowB));
                    }
                }
                if (m1 < a.M) {
                    a.y[(size_t)m1 * a.N + rowA] = a1;
                    a.y[(size_t)m1 * a.N + rowB] = b1;
                    if (ARGMAX) {
                        atomicMax(&ck[m1], argmax_key(a1, (uint32_t)rowA));
                        atomicMax(&ck[m1], argmax_key(b1, (uint32_t)rowB));
                    }
                }
                a0 = a1 = b0 = b1 = 0.f;
            }
        }
    };
    if (f16)
        run(std::true_type{});
    else
        run(std::false_type{});

    if (failed >= 0 && lane == 0)
        for (int f = failed; f < issued; ++f)
            mbar_wait_bounded(bar0 + 8u * (f % kSlots), (uint32_t)((f / kSlots) & 1), kDrainLimit);
    __syncthreads();
    if (ARGMAX && threadIdx.x < a.M)
        a.keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = ck[threadIdx.x];
}

} // namespace

// Tensor maps of the slot kernels: codes as uint32 {32 words, K/256 lines,
// N rows} with box {32, lines, 16} and the 128-byte swizzle; with steps != null
// also the group-32 steps as uint16 {K/32, N} with box {steps_box, 16} (its row
// stride K/16 bytes is a multiple of 16 since K % 256 == 0; the callers check
// that the base is 16-byte aligned).
static bool encode_slot_maps(CUtensorMap *codes, CUtensorMap *steps, const uint32_t *qw, const uint16_t *sc, int N,
                             int K, int lines, int steps_box)
{
    auto enc = tmap_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {32, (cuuint64_t)(K / 256), (cuuint64_t)N};
    cuuint64_t strides[2] = {128, (cuuint64_t)K / 2};
    cuuint32_t box[3] = {32, (cuuint32_t)lines, 16};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t *>(qw), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (steps == nullptr)
        return true;
    cuuint64_t sd[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
    cuuint64_t ss[1] = {(cuuint64_t)K / 16};
    cuuint32_t sbx[2] = {(cuuint32_t)steps_box, 16};
    cuuint32_t ses[2] = {1, 1};
    return enc(steps, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(sc), sd, ss, sbx, ses,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool vocab_supported(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc)
{
    const int nrb = N / 16;
    // Group 32 takes its steps by tensor copy (16-byte aligned steps); larger
    // groups share one step per lane pair and load it from global memory.
    // At least two slots per row block (K >= 1536): with one, a warp has too few
    // fills to keep a copy in flight (80560 x 768 measured slower).
    return M == 1 && K % (kTs * 128) == 0 && K >= 2 * kTs * 128 && N % 16 == 0 && nrb >= 2 * num_sms * kWarps &&
           (reinterpret_cast<uintptr_t>(qw) & 15) == 0 && (lg > 0 || (reinterpret_cast<uintptr_t>(sc) & 15) == 0) &&
           tmap_encoder() != nullptr &&
           kSmem + (size_t)kWarps * kSlots * kStepBytes + (size_t)K * 2 + 64 + 1024 <= 226 * 1024;
}

cudaError_t run_decode_vocab(float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int N, int K,
                             int lg, unsigned long long *keys, int32_t *argmax, int *err, int num_sms,
                             cudaStream_t s, const int32_t *forced)
{
    // Codes {32, 3, 16} boxes; steps by tensor copy only at group 32 (a steps
    // row of K/group bf16 is not always a multiple of 16 bytes otherwise).
    const bool g32_tma = lg == 0;
    CUtensorMap map, smap;
    if (!encode_slot_maps(&map, g32_tma ? &smap : nullptr, qw, sc, N, K, kLines, kTs * 4))
        return cudaErrorInvalidValue;
    if (!g32_tma)
        smap = map;
    VocabArgs a;
    a.y = y;
    a.x = x;
    a.sc = sc;
    a.keys = keys;
    a.err = err;
    a.forced = argmax != nullptr ? forced : nullptr;
    a.N = N;
    a.K = K;
    a.lg = lg;
    const size_t smem = kSmem + (g32_tma ? (size_t)kWarps * kSlots * kStepBytes : 0) + (size_t)(K / 8 + 8) * 16 + 1024;
    const bool am = argmax != nullptr;
    auto kern = am ? (g32_tma ? w4_decode_vocab_kernel<true, true> : w4_decode_vocab_kernel<true, false>)
                   : (g32_tma ? w4_decode_vocab_kernel<false, true> : w4_decode_vocab_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, map, smap);
    if (e != cudaSuccess || !am)
        return e;
    return run_argmax_finalize(argmax, keys, 1, num_sms, s, a.forced);
}

// Shared memory of the slab form for W warps (x rows: 2 when rotated), and the
// warp count it launches with: 16 when that fits (and the units fill the
// slots), else 8; 0 if neither holds every unit within the slots.
static size_t slab_smem(int W, int R, int S, int K, bool rot)
{
    return (size_t)W * kSlots * (kSlotBytes + kStepBytes) + (size_t)((rot ? 2 : 1) * (K / 8) + 8) * 16 +
           (size_t)R * S * 16 * 4 + 1024;
}

static int slab_warps(int R, int S, int K, bool rot)
{
    for (int W = kWarps; W >= 8; W /= 2)
        if (R * S <= W * kSlots && slab_smem(W, R, S, K, rot) <= 226 * 1024)
            return W;
    return 0;
}

// Row blocks per CTA of the slab form and whether it serves (N, K): group 32,
// K % 768 == 0, N % 16 == 0, 16-byte aligned codes and steps, a CTA's units
// within its 32 slots (so every copy is issued before the dependency wait),
// below vocabulary sizes; hblock (256 or 512): rotated weights.
int slab_rows_per_cta(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc, int hblock)
{
    if (M != 1 || lg != 0 || K % (kTs * 128) != 0 || N % 16 != 0 || num_sms < 1)
        return 0;
    if (hblock != 0 && ((hblock != 256 && hblock != 512) || K % hblock != 0))
        return 0;
    if ((reinterpret_cast<uintptr_t>(qw) & 15) != 0 || (reinterpret_cast<uintptr_t>(sc) & 15) != 0 ||
        tmap_encoder() == nullptr)
        return 0;
    const int nrb = N / 16, S = K / (kTs * 128);
    const int R = (nrb + num_sms - 1) / num_sms;
    if (nrb >= 2 * num_sms * kWarps || slab_warps(R, S, K, hblock != 0) == 0)
        return 0;
    return R;
}

cudaError_t run_decode_slab(int R, float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int N,
                            int K, int *err, cudaStream_t s, int hblock)
{
    if (R < 1)
        return cudaErrorNotSupported;
    CUtensorMap map, smap;
    if (!encode_slot_maps(&map, &smap, qw, sc, N, K, kLines, kTs * 4))
        return cudaErrorInvalidValue;
    VocabArgs a;
    a.y = y;
    a.x = x;
    a.sc = sc;
    a.keys = nullptr;
    a.err = err;
    a.forced = nullptr;
    a.N = N;
    a.K = K;
    a.lg = 0;
    const bool rot = hblock != 0;
    const int S = K / (kTs * 128), nrb = N / 16;
    const int W = slab_warps(R, S, K, rot);
    if (W == 0)
        return cudaErrorNotSupported;
    const size_t smem = slab_smem(W, R, S, K, rot);
    auto kern = !rot ? w4_decode_slab_kernel<0>
                     : (hblock == 256 ? w4_decode_slab_kernel<8> : w4_decode_slab_kernel<16>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((nrb + R - 1) / R);
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const float norm = rot ? 1.0f / sqrtf((float)hblock) : 0.f;
    return cudaLaunchKernelEx(&cfg, kern, a, R, norm, map, smap);
}

// ------------------------------------------------------------ M <= 8 ----

// Shared memory of the M <= 8 slot form with W warps.
static size_t slots8_smem(int W, int M, int K)
{
    return (size_t)W * kSlots * (kSlotBytes + kStepBytes) + (size_t)M * (K / 8) * 16 + 16 * 16 + 1024;
}

Slots8Plan plan_slots8(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc)
{
    Slots8Plan p;
    if (M < 2 || M > 8 || lg != 0 || K % (kTs * 128) != 0 || N % 16 != 0 || num_sms < 1)
        return p;
    if ((reinterpret_cast<uintptr_t>(qw) & 15) != 0 || (reinterpret_cast<uintptr_t>(sc) & 15) != 0 ||
        tmap_encoder() == nullptr)
        return p;
    // As many warps as the shared memory holds; every warp of the wave walks
    // at least two row blocks.
    int W = kWarps;
    while (W >= 4 && slots8_smem(W, M, K) > 226 * 1024)
        --W;
    if (W < 4 || N / 16 < 2 * num_sms * W)
        return p;
    p.ok = true;
    p.W = W;
    p.grid = num_sms;
    p.smem = slots8_smem(W, M, K);
    return p;
}

cudaError_t run_decode_slots8(const Slots8Plan &p, float *y, const uint16_t *x, const uint32_t *qw,
                              const uint16_t *sc, int M, int N, int K, unsigned long long *keys, int32_t *argmax,
                              int *err, cudaStream_t s)
{
    if (!p.ok)
        return cudaErrorNotSupported;
    CUtensorMap map, smap;
    if (!encode_slot_maps(&map, &smap, qw, sc, N, K, kLines, kTs * 4))
        return cudaErrorInvalidValue;
    Slots8Args a;
    a.y = y;
    a.x = x;
    a.keys = keys;
    a.err = err;
    a.M = M;
    a.N = N;
    a.K = K;
    const bool am = argmax != nullptr;
    auto kern = am ? w4_decode_slots8_kernel<true> : w4_decode_slots8_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.W * 32);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, map, smap);
    if (e != cudaSuccess || !am)
        return e;
    return run_argmax_finalize(argmax, keys, M, p.grid, s);
}

} // namespace w4
