// Decode-form W4A16 GEMV/GEMM (M = 1..8) on the warp-level tensor core.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
// (decode multiplies one vector by every weight matrix, so the speed limit is
// reading the weights; the kernel reads the packed 4-bit words, unpacks them in
// registers and multiplies, never writing a 16-bit copy) and the tiling
// paragraph (each weight shape gets its own fixed tiling).
//
// GB300 design. At ~6.8 TB/s and 0.5625 B per weight the kernel must consume
// ~12e12 weights/s, i.e. ~3 lane-instructions per weight at 2 GHz over 152 SMs.
// A CUDA-core dot product (unpack + convert + FMA per weight) does not fit, so
// every 16x16 block of exact (code - 8) values goes to one m16n8k16 bf16 mma
// with fp32 accumulation; the unpack is ~1.4 instructions per weight.
// The group step is applied in fp32 after the mma, per group, which keeps the
// result within 1e-4 of the exact sum (no bf16 rounding of weights).
//
// Kernel "m2" (M = 1 or 2): lane (g, t) of a warp loads one full group (32
// codes, 16 B) of rows g and g+8, group 4*kt + t of k-tile kt, with one 128-bit
// load each. The four lanes of a quad therefore hold four different groups, and
// the mma's eight B columns separate them: column 4*m + s carries x-row m
// restricted to group-slot s (zero elsewhere). After the 8 mmas of a k-tile,
// C[row][4m+s] is the unscaled partial of (row, group 4kt+s, x-row m), which is
// scaled in fp32 and accumulated.
//
// Kernel "m8" (M = 3..8): lane (g, t) loads word t of one group for rows g and
// g+8 (32-bit loads); B columns are the x rows; one group per two mmas.
//
// Both kernels issue their first weight loads (and an L2 prefetch of x) before
// griddepcontrol.wait, so under programmatic dependent launch the weight
// stream of this call overlaps the tail of the previous kernel; x is read into
// the SM only after the wait. Measured on GB300 inside a graph-replayed decode
// sweep, the time after the wait is latency, not bandwidth: the x round trip
// and the per-warp chain of dependent mmas. Hence small shapes split K finely
// (one to three k-tiles per warp, up to 16 warps per row block), x is staged
// with all of a thread's loads in flight at once, and the 8 mmas of a k-tile
// accumulate into two independent chains.
#include "common.cuh"
#include "internal.h"

#include <atomic>
#include <mutex>

namespace w4 {

static constexpr int kTileK = 128; // k per tile of the m2 kernel: 4 groups
// Shared memory two resident CTAs of the persistent forms may take together
// (228 KB per SM, less 1 KB reserved per CTA and some headroom).
static constexpr size_t kSmemPerSm = 220 * 1024;

// xs[m * cpr + c] = permute_x8(x[m][8c .. 8c+7]) for m < rows, c < cpr (chunks
// at or past K/8 are zero). Each thread issues up to kXLoads loads before it
// uses any, so the staging costs one memory round trip, not one per chunk.
__device__ __forceinline__ void stage_x_rows(uint4 *xs, const uint16_t *x, int rows, int K, int cpr)
{
    constexpr int kXLoads = 4;
    const int total = rows * cpr, kc = K >> 3;
    for (int i0 = threadIdx.x; i0 < total; i0 += kXLoads * blockDim.x) {
        uint4 v[kXLoads];
#pragma unroll
        for (int j = 0; j < kXLoads; ++j) {
            const int i = i0 + j * blockDim.x;
            const int m = i / cpr, c = i - m * cpr;
            v[j] = (i < total && c < kc) ? *reinterpret_cast<const uint4 *>(x + (size_t)m * K + c * 8)
                                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < kXLoads; ++j) {
            const int i = i0 + j * blockDim.x;
            if (i < total)
                xs[i] = permute_x8(v[j]);
        }
    }
}

// The steps of the 32-code groups j and j + 1 (j even) of one row. Rows hold
// one step per 32 << lg codes. G32 (lg == 0): the two steps as a bf16 pair, low
// half first. Otherwise (lg >= 1, the only case the !G32 kernels are launched
// for) both groups share one step, returned in the low half; the kernels then
// scale the sum of the two groups' products with it (one FMA instead of two and
// no duplicated step: 6-7% faster at group 256 on the M = 1 sweep shapes).
template <bool G32>
__device__ __forceinline__ uint32_t step_pair(const uint16_t *srow, int j, int lg)
{
    if (G32)
        return ldg_nc_u32(srow + j);
    return ldg_nc_u16(srow + (j >> lg));
}

// The M <= 8 kernels' x staging (cpr == K / 8, every chunk real): all of a
// thread's chunks in flight at once as asynchronous 16-byte copies, then the
// pair permutation in place, each thread permuting the chunks it copied (its
// own completed copies are visible to it, so no barrier sits between the two
// passes); the caller synchronises before use. At M = 8 and
// large K a thread stages up to 24 chunks, which the register path above
// would fetch in six dependent round trips (measured on GB300: the M = 8
// sweep 0.89 -> 0.82 ms, every shape faster in the sweep).
__device__ __forceinline__ void stage_x_rows_async(uint4 *xs, const uint16_t *x, int rows, int K)
{
    const int total = rows * (K >> 3);
    const uint32_t base = smem_addr(xs);
    for (int i = threadIdx.x; i < total; i += blockDim.x)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + 16u * (uint32_t)i),
                     "l"(x + 8 * (size_t)i)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    for (int i = threadIdx.x; i < total; i += blockDim.x)
        xs[i] = permute_x8(xs[i]);
}

// ---------------------------------------------------------------- m2 ----

// FULL (K % 128 == 0, implies SC32): every k-tile is whole, so the loads need
// no per-group guards; warps past the last row block load clamped rows and
// never store.
// PAIRS: x rows come as (hi, lo) pairs of one activation row (the two bf16
// parts of an fp32 value); each output row is the sum of its pair.
template <int MX, int U, bool SC32, bool FULL, bool ARGMAX, bool G32, bool PAIRS>
__global__ void __launch_bounds__(512)
w4_decode_m2_kernel(float *__restrict__ y, const uint16_t *__restrict__ x,
               const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc,
               int N, int K, int ksplit, unsigned long long *__restrict__ keys, int lg,
               const int32_t *__restrict__ forced, int hb, float hnorm)
{
    extern __shared__ __align__(16) unsigned char smem[];
    if (ARGMAX && forced != nullptr && *forced >= 0) {
        // The next token is forced: no weight is read (finalize writes it).
        pdl_launch_dependents();
        pdl_wait();
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nwarps = blockDim.x >> 5;
    const int rbc = nwarps / ksplit;
    const int ks = warp % ksplit, rbl = warp / ksplit;
    const int nrb = (N + 15) >> 4;
    const int rb = blockIdx.x * rbc + rbl;
    const bool active = rb < nrb;
    const int T = (K + kTileK - 1) / kTileK;
    const int ngroups = K >> 5;
    const int Kpad = T * kTileK;
    const int kt0 = (int)((long long)T * ks / ksplit);
    const int nkt = (int)((long long)T * (ks + 1) / ksplit) - kt0;

    const int rowA = rb * 16 + g, rowB = rowA + 8;
    const int rA = min(rowA, N - 1), rB = min(rowB, N - 1);
    const uint32_t *qA = qw + (size_t)rA * (K >> 3) + 4 * t;
    const uint32_t *qB = qw + (size_t)rB * (K >> 3) + 4 * t;
    // Steps: one per 32 << lg codes, K >> (5 + lg) per row. This lane scales
    // the 32-code groups 4kt + jt and 4kt + jt + 1 (one pair).
    const int sstride = G32 ? ngroups : (ngroups >> lg);
    const uint16_t *sA = sc + (size_t)rA * sstride;
    const uint16_t *sB = sc + (size_t)rB * sstride;
    const int jt = 2 * (t & 1);
    const uint16_t *sAj = sA + jt, *sBj = sB + jt; // group 32: this lane's pair

    uint4 wa[U], wb[U];
    uint32_t sa[U], sb[U];

    auto load = [&](int u, int kt) {
        if (FULL) {
            wa[u] = ldg_stream_v4(qA + 16 * kt);
            wb[u] = ldg_stream_v4(qB + 16 * kt);
            if (G32) {
                sa[u] = ldg_nc_u32(sAj + 4 * kt);
                sb[u] = ldg_nc_u32(sBj + 4 * kt);
            } else {
                sa[u] = step_pair<false>(sA, 4 * kt + jt, lg);
                sb[u] = step_pair<false>(sB, 4 * kt + jt, lg);
            }
            return;
        }
        const int G = 4 * kt + t;
        if (active && G < ngroups) {
            wa[u] = ldg_stream_v4(qA + 16 * kt);
            wb[u] = ldg_stream_v4(qB + 16 * kt);
        } else {
            wa[u] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
            wb[u] = wa[u];
        }
        const int Gs = 4 * kt + 2 * (t & 1);
        if (SC32) {
            const bool ok = active && Gs < ngroups;
            sa[u] = ok ? step_pair<G32>(sA, Gs, lg) : 0u;
            sb[u] = ok ? step_pair<G32>(sB, Gs, lg) : 0u;
        } else { // K % 64 != 0, so the group is 32 (lg == 0)
            const bool ok0 = active && Gs < ngroups, ok1 = active && Gs + 1 < ngroups;
            sa[u] = (ok0 ? ldg_nc_u16(sA + Gs) : 0u) | ((ok1 ? ldg_nc_u16(sA + Gs + 1) : 0u) << 16);
            sb[u] = (ok0 ? ldg_nc_u16(sB + Gs) : 0u) | ((ok1 ? ldg_nc_u16(sB + Gs + 1) : 0u) << 16);
        }
    };

    // Stream the first weight tiles before waiting on the previous kernel.
    // (hb > 0: x is one row that this kernel rotates into the pair rows.)
    const bool fused = PAIRS && hb > 0;
    if (threadIdx.x == 32)
        prefetch_l2_bulk(x, (uint32_t)((fused ? 1 : MX) * K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < nkt)
            load(u, kt0 + u);
    pdl_launch_dependents();
    pdl_wait();

    // Stage x, permuted into the B-operand pair order, and a zero chunk.
    uint4 *xs = reinterpret_cast<uint4 *>(smem);
    const int chunks_per_row = Kpad >> 3;
    uint4 *zero_chunk = xs + MX * chunks_per_row;
    if (fused) {
        if (hb == 256)
            stage_x_hadamard<8>(xs, x, K, chunks_per_row, hnorm);
        else
            stage_x_hadamard<16>(xs, x, K, chunks_per_row, hnorm);
    } else {
        stage_x_rows(xs, x, MX, K, chunks_per_row);
    }
    if (threadIdx.x == 0)
        *zero_chunk = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // This lane feeds B column g: x-row g>>2 restricted to group-slot g&3,
    // which lives on lanes with t == g&3.
    const int bm = g >> 2;
    const bool bsel = ((g & 3) == t) && (bm < MX);
    const uint4 *xrow = bsel ? xs + bm * chunks_per_row + 4 * t : zero_chunk;
    const int xstep = bsel ? 16 : 0; // chunks per k-tile
    const int xi = bsel ? 1 : 0;     // chunk stride between words

    float accA = 0.f, accB = 0.f;

    auto compute = [&](int u, int kt) {
        // Two independent accumulator chains (4 mmas each) instead of one of 8.
        float c[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 *xb = xrow + xstep * kt;
        const uint32_t a_w[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        const uint32_t b_w[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 b = xb[xi * i];
            unpack_mma2(c, d, a_w[i], b_w[i], b.x, b.y, b.z, b.w);
        }
        if (G32) {
            accA = fmaf(bf16lo_to_f32(sa[u]), c[0] + d[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u]), c[1] + d[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), c[2] + d[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u]), c[3] + d[3], accB);
        } else { // one step for both groups
            accA = fmaf(bf16lo_to_f32(sa[u]), (c[0] + d[0]) + (c[1] + d[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), (c[2] + d[2]) + (c[3] + d[3]), accB);
        }
    };

    // Two tiles at once (four independent mma chains, twice the independent
    // unpack work between dependent instructions); the same sums in the same
    // order as one tile at a time.
    auto compute2 = [&](int u, int kt) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, d0[4] = {0.f, 0.f, 0.f, 0.f};
        float c1[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 *xb = xrow + xstep * kt;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 b0 = xb[xi * i], b1 = xb[xstep + xi * i];
            unpack_mma2(c0, d0, (&wa[u].x)[i], (&wb[u].x)[i], b0.x, b0.y, b0.z, b0.w);
            unpack_mma2(c1, d1, (&wa[u + 1].x)[i], (&wb[u + 1].x)[i], b1.x, b1.y, b1.z, b1.w);
        }
        if (G32) {
            accA = fmaf(bf16lo_to_f32(sa[u]), c0[0] + d0[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u]), c0[1] + d0[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), c0[2] + d0[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u]), c0[3] + d0[3], accB);
            accA = fmaf(bf16lo_to_f32(sa[u + 1]), c1[0] + d1[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u + 1]), c1[1] + d1[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u + 1]), c1[2] + d1[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u + 1]), c1[3] + d1[3], accB);
        } else {
            accA = fmaf(bf16lo_to_f32(sa[u]), (c0[0] + d0[0]) + (c0[1] + d0[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), (c0[2] + d0[2]) + (c0[3] + d0[3]), accB);
            accA = fmaf(bf16lo_to_f32(sa[u + 1]), (c1[0] + d1[0]) + (c1[1] + d1[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u + 1]), (c1[2] + d1[2]) + (c1[3] + d1[3]), accB);
        }
    };

    // Measured on GB300 in the graph-replayed decode sweep: pairs pay where a
    // warp's tiles are all preloaded (1536 x 12288: 5.50 -> 5.39 us) and lose
    // where tiles are refilled, since a pair delays its two refills
    // (24576 x 1536: 6.95 -> 7.82 us).
    if (U == 8 && MX == 1 && nkt <= U) {
#pragma unroll
        for (int u = 0; u < U; u += 2) {
            if (u + 1 < nkt)
                compute2(u, kt0 + u);
            else if (u < nkt)
                compute(u, kt0 + u);
        }
    } else {
        for (int base = 0; base < nkt; base += U) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (base + u < nkt) {
                    compute(u, kt0 + base + u);
                    if (base + u + U < nkt)
                        load(u, kt0 + base + u + U);
                }
            }
        }
    }

    // Lanes t and t^1 hold the two group-slot pairs of the same (row, x-row).
    accA += __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
    accB += __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
    if (PAIRS) { // x-rows 0 (lanes t < 2) and 1 (t >= 2) are one output row
        accA += __shfl_xor_sync(0xFFFFFFFFu, accA, 2);
        accB += __shfl_xor_sync(0xFFFFFFFFu, accB, 2);
    }
    constexpr int MO = PAIRS ? MX / 2 : MX; // output rows
    const int m = t >> 1;
    const bool writer = ((t & 1) == 0) && (m < MO);

    __shared__ unsigned long long ck[MO];
    if (ARGMAX) {
        if (threadIdx.x < MO)
            ck[threadIdx.x] = 0ull;
        __syncthreads();
    }

    if (ksplit == 1) {
        if (writer && active) {
            if (rowA < N) {
                y[(size_t)m * N + rowA] = accA;
                if (ARGMAX)
                    atomicMax(&ck[m], argmax_key(accA, rowA));
            }
            if (rowB < N) {
                y[(size_t)m * N + rowB] = accB;
                if (ARGMAX)
                    atomicMax(&ck[m], argmax_key(accB, rowB));
            }
        }
    } else {
        // Fixed-order reduction of the k-slices through shared memory.
        float *red = reinterpret_cast<float *>(zero_chunk + 1); // [rbc][ksplit][MO][16]
        if (writer) {
            float *r = red + ((rbl * ksplit + ks) * MO + m) * 16;
            r[g] = accA;
            r[g + 8] = accB;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < rbc * MO * 16; i += blockDim.x) {
            const int rr = i & 15, mm = (i >> 4) % MO, rl = i / (16 * MO);
            const int row = (blockIdx.x * rbc + rl) * 16 + rr;
            float s = 0.f;
            for (int k2 = 0; k2 < ksplit; ++k2)
                s += red[((rl * ksplit + k2) * MO + mm) * 16 + rr];
            if (row < N) {
                y[(size_t)mm * N + row] = s;
                if (ARGMAX)
                    atomicMax(&ck[mm], argmax_key(s, row));
            }
        }
    }

    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x < MO)
            keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = ck[threadIdx.x];
    }
}

// ------------------------------------------------------- persistent m2 ----
//
// Large N (the vocabulary projection): two resident CTAs of 8 warps per SM,
// each warp owning every (grid*8)-th 16-row block (ks = 1, whole rows), its
// k-tiles flattened into one stream so that the 8 tiles in flight run on across
// row-block boundaries instead of draining and refilling every block (one wave
// instead of ~7). K % 256 == 0 and N % 16 == 0. Loads walk running pointers,
// and k-tiles are computed in pairs (four independent mma chains): measured
// 59.0 -> 48.9 us for a 262144 x 1536 GEMV against one tile at a time with
// addresses recomputed per load; 4 tiles in flight per warp (105 registers)
// then beat 6, 8 or 12 (46.3 vs 48.1, 49.0, 63.0 us) and 3 or 4 CTAs per SM.
template <int MX, int U, int MINB, bool ARGMAX, bool G32, bool PAIRS>
__global__ void __launch_bounds__(256, MINB)
w4_decode_m2_persist_kernel(float *__restrict__ y, const uint16_t *__restrict__ x,
                       const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc, int N, int K,
                       unsigned long long *__restrict__ keys, int lg, const int32_t *__restrict__ forced,
                       int hb, float hnorm)
{
    extern __shared__ __align__(16) unsigned char smem[];
    if (ARGMAX && forced != nullptr && *forced >= 0) {
        pdl_launch_dependents();
        pdl_wait();
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nrb = (N + 15) >> 4;
    const int T = K / kTileK;
    const int ngroups = K >> 5;
    const int GW = gridDim.x * 8, gw = blockIdx.x * 8 + warp;
    const int nmine = nrb > gw ? (nrb - gw + GW - 1) / GW : 0;
    const int Q = nmine * T; // k-tiles of this warp, row block by row block

    uint4 wa[U], wb[U];
    uint32_t sa[U], sb[U];
    // Loader pointers (N % 16 == 0: no clamped rows): row A of the warp's
    // current row block at its current k-tile; row B is 8 rows (K words) on.
    const uint32_t *lp = qw + (size_t)(gw * 16 + g) * (K >> 3) + 4 * t;
    // Step row of row A and this lane's 32-code group index in it (steps: one
    // per 32 << lg codes).
    const int sstride = ngroups >> lg;
    const uint16_t *ls = sc + (size_t)(gw * 16 + g) * sstride;
    int lj = 2 * (t & 1);
    const size_t rb_words = (size_t)GW * 16 * (K >> 3) - (size_t)16 * T;
    const size_t rb_steps = (size_t)GW * 16 * sstride;
    const size_t rowB_steps = (size_t)8 * sstride;
    int lkt = 0;
    auto load = [&](int u) {
        wa[u] = ldg_stream_v4(lp);
        wb[u] = ldg_stream_v4(lp + K);
        sa[u] = step_pair<G32>(ls, lj, lg);
        sb[u] = step_pair<G32>(ls + rowB_steps, lj, lg);
        lp += 16;
        lj += 4;
        if (++lkt == T) {
            lkt = 0;
            lp += rb_words;
            ls += rb_steps;
            lj = 2 * (t & 1);
        }
    };

    const bool fused = PAIRS && hb > 0; // x is one row, rotated here into the pair rows
    if (threadIdx.x == 32)
        prefetch_l2_bulk(x, (uint32_t)((fused ? 1 : MX) * K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < Q)
            load(u);
    pdl_launch_dependents();
    pdl_wait();

    uint4 *xs = reinterpret_cast<uint4 *>(smem);
    const int chunks_per_row = K >> 3;
    uint4 *zero_chunk = xs + MX * chunks_per_row;
    if (fused) {
        if (hb == 256)
            stage_x_hadamard<8>(xs, x, K, chunks_per_row, hnorm);
        else
            stage_x_hadamard<16>(xs, x, K, chunks_per_row, hnorm);
    } else {
        stage_x_rows(xs, x, MX, K, chunks_per_row);
    }
    constexpr int MO = PAIRS ? MX / 2 : MX; // output rows (PAIRS: x-rows 0, 1 are one)
    __shared__ unsigned long long ck[MO];
    if (threadIdx.x == 0)
        *zero_chunk = make_uint4(0u, 0u, 0u, 0u);
    if (ARGMAX && threadIdx.x < MO)
        ck[threadIdx.x] = 0ull;
    __syncthreads();

    const int bm = g >> 2;
    const bool bsel = ((g & 3) == t) && (bm < MX);
    const uint4 *xrow = bsel ? xs + bm * chunks_per_row + 4 * t : zero_chunk;
    const int xstep = bsel ? 16 : 0;
    const int xi = bsel ? 1 : 0;
    const int m = t >> 1;
    const bool writer = ((t & 1) == 0) && (m < MO);

    float accA = 0.f, accB = 0.f;
    int cj = 0, ckt = 0; // compute cursor
    // Two consecutive k-tiles of the same row block at once: four independent
    // mma chains and twice the independent unpack work per step.
    auto compute2 = [&](int u) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, d0[4] = {0.f, 0.f, 0.f, 0.f};
        float c1[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 *xb = xrow + xstep * ckt;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 b0 = xb[xi * i], b1 = xb[xstep + xi * i];
            unpack_mma2(c0, d0, (&wa[u].x)[i], (&wb[u].x)[i], b0.x, b0.y, b0.z, b0.w);
            unpack_mma2(c1, d1, (&wa[u + 1].x)[i], (&wb[u + 1].x)[i], b1.x, b1.y, b1.z, b1.w);
        }
        if (G32) {
            accA = fmaf(bf16lo_to_f32(sa[u]), c0[0] + d0[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u]), c0[1] + d0[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), c0[2] + d0[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u]), c0[3] + d0[3], accB);
            accA = fmaf(bf16lo_to_f32(sa[u + 1]), c1[0] + d1[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u + 1]), c1[1] + d1[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u + 1]), c1[2] + d1[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u + 1]), c1[3] + d1[3], accB);
        } else { // one step for both groups
            accA = fmaf(bf16lo_to_f32(sa[u]), (c0[0] + d0[0]) + (c0[1] + d0[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), (c0[2] + d0[2]) + (c0[3] + d0[3]), accB);
            accA = fmaf(bf16lo_to_f32(sa[u + 1]), (c1[0] + d1[0]) + (c1[1] + d1[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u + 1]), (c1[2] + d1[2]) + (c1[3] + d1[3]), accB);
        }
    };
    auto finish = [&]() {
        float a = accA + __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
        float b = accB + __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
        if (PAIRS) {
            a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
            b += __shfl_xor_sync(0xFFFFFFFFu, b, 2);
        }
        const int rowA = (gw + cj * GW) * 16 + g, rowB = rowA + 8;
        if (writer) {
            if (rowA < N) {
                y[(size_t)m * N + rowA] = a;
                if (ARGMAX)
                    atomicMax(&ck[m], argmax_key(a, rowA));
            }
            if (rowB < N) {
                y[(size_t)m * N + rowB] = b;
                if (ARGMAX)
                    atomicMax(&ck[m], argmax_key(b, rowB));
            }
        }
        accA = accB = 0.f;
    };

    // T is even, so a pair never straddles two row blocks.
    for (int base = 0; base < Q; base += U) {
#pragma unroll
        for (int u = 0; u < U; u += 2) {
            if (base + u < Q) {
                compute2(u);
                if (base + u + U < Q) {
                    load(u);
                    load(u + 1);
                }
                ckt += 2;
                if (ckt == T) {
                    finish();
                    ckt = 0;
                    ++cj;
                }
            }
        }
    }

    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x < MO)
            keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = ck[threadIdx.x];
    }
}

// ---------------------------------------------------------------- m8 ----

// 4x4 transpose of 32-bit words across the four lanes of a quad: lane t holds
// v[j] = W[t][j] on entry and W[j][t] on return (t = lane & 3). Two exchange
// stages (lane bit 1 with register bit 1, then bit 0 with bit 0), one shuffle
// per register pair and stage.
__device__ __forceinline__ void quad_transpose4(uint32_t (&v)[4], int t)
{
#pragma unroll
    for (int bit = 1; bit >= 0; --bit) {
        const int m = 1 << bit;
        const bool hi = (t >> bit) & 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j & m)
                continue;
            const int jj = j | m;
            const uint32_t send = hi ? v[j] : v[jj];
            const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, m);
            if (hi)
                v[j] = recv;
            else
                v[jj] = recv;
        }
    }
}

// Output of the M <= 8 kernels: lane (g, t) holds y[2t][rowA], y[2t+1][rowA],
// y[2t][rowB], y[2t+1][rowB] of its warp's K slice; with ksplit > 1 the slices
// are added in fixed order through shared memory (red: [rbc][ksplit][8][16]).
// PAIRS: x-rows 2t and 2t+1 are the two parts of output row t (M/2 outputs).
// CTA-best argmax key per output row; max is order-independent (deterministic).
template <bool ARGMAX, bool PAIRS>
__device__ __forceinline__ void m8_store(float *__restrict__ y, float a0, float a1, float b0, float b1,
                                         int M, int N, int g, int t, int rowA, int rowB, bool active,
                                         int ksplit, int ks, int rbl, int rbc, float *red,
                                         unsigned long long *__restrict__ keys)
{
    __shared__ unsigned long long ck[8];
    if (ARGMAX) {
        if (threadIdx.x < 8)
            ck[threadIdx.x] = 0ull;
        __syncthreads();
    }
    if (PAIRS) {
        a0 += a1;
        b0 += b1;
    }
    const int Mout = PAIRS ? M / 2 : M;
    const int m0 = PAIRS ? t : 2 * t, m1 = 2 * t + 1;
    constexpr int NJ = PAIRS ? 1 : 2;
    if (ksplit == 1) {
        if (active) {
            const float v[2][2] = {{a0, a1}, {b0, b1}};
            const int rows[2] = {rowA, rowB};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int mm = j ? m1 : m0;
                    if (rows[h] < N && mm < Mout) {
                        y[(size_t)mm * N + rows[h]] = v[h][j];
                        if (ARGMAX)
                            atomicMax(&ck[mm], argmax_key(v[h][j], rows[h]));
                    }
                }
            }
        }
    } else {
        float *r = red + (rbl * ksplit + ks) * 8 * 16;
        r[m0 * 16 + g] = a0;
        r[m0 * 16 + g + 8] = b0;
        if (!PAIRS) {
            r[m1 * 16 + g] = a1;
            r[m1 * 16 + g + 8] = b1;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < rbc * 8 * 16; i += blockDim.x) {
            const int rr = i & 15, mm = (i >> 4) & 7, rl = i >> 7;
            const int row = (blockIdx.x * rbc + rl) * 16 + rr;
            if (row < N && mm < Mout) {
                float sum = 0.f;
                for (int k2 = 0; k2 < ksplit; ++k2)
                    sum += red[((rl * ksplit + k2) * 8 + mm) * 16 + rr];
                y[(size_t)mm * N + row] = sum;
                if (ARGMAX)
                    atomicMax(&ck[mm], argmax_key(sum, row));
            }
        }
    }
    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x < Mout)
            keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = ck[threadIdx.x];
    }
}

template <int U, bool ARGMAX, bool PAIRS>
__global__ void __launch_bounds__(512)
w4_decode_m8_kernel(float *__restrict__ y, const uint16_t *__restrict__ x,
               const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc,
               int M, int N, int K, int ksplit, unsigned long long *__restrict__ keys, int lg)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nwarps = blockDim.x >> 5;
    const int rbc = nwarps / ksplit;
    const int ks = warp % ksplit, rbl = warp / ksplit;
    const int nrb = (N + 15) >> 4;
    const int rb = blockIdx.x * rbc + rbl;
    const bool active = rb < nrb;
    const int ngroups = K >> 5;
    const int G0 = (int)((long long)ngroups * ks / ksplit);
    const int nG = (int)((long long)ngroups * (ks + 1) / ksplit) - G0;

    const int rowA = rb * 16 + g, rowB = rowA + 8;
    const int rA = min(rowA, N - 1), rB = min(rowB, N - 1);
    const uint32_t *qA = qw + (size_t)rA * (K >> 3) + t;
    const uint32_t *qB = qw + (size_t)rB * (K >> 3) + t;
    const uint16_t *sA = sc + (size_t)rA * (ngroups >> lg);
    const uint16_t *sB = sc + (size_t)rB * (ngroups >> lg);

    uint32_t wa[U], wb[U], sa[U], sb[U];
    auto load = [&](int u, int G) {
        if (active) {
            wa[u] = ldg_stream_u32(qA + 4 * G);
            wb[u] = ldg_stream_u32(qB + 4 * G);
            sa[u] = ldg_nc_u16(sA + (G >> lg));
            sb[u] = ldg_nc_u16(sB + (G >> lg));
        } else {
            wa[u] = wb[u] = 0x88888888u;
            sa[u] = sb[u] = 0u;
        }
    };

    if (threadIdx.x == 32)
        prefetch_l2_bulk(x, (uint32_t)(M * K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < nG)
            load(u, G0 + u);
    pdl_launch_dependents();
    pdl_wait();

    uint4 *xs = reinterpret_cast<uint4 *>(smem); // [8][K/8] permuted chunks
    const int cpr = K >> 3;
    stage_x_rows_async(xs, x, M, K);
    if (M < 8) // rows M..7 of the B operand are zero
        for (int i = M * cpr + threadIdx.x; i < 8 * cpr; i += blockDim.x)
            xs[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // B column g is x-row g; this lane supplies word t of each group.
    const uint4 *xrow = xs + g * cpr + t;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;

    auto compute = [&](int u, int G) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 bx = xrow[4 * G];
        uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
        unpack_word(wa[u], a04, a15, a26, a37);
        unpack_word(wb[u], b04, b15, b26, b37);
        mma_16816(c, a04, b04, a15, b15, bx.x, bx.y);
        mma_16816(c, a26, b26, a37, b37, bx.z, bx.w);
        const float s_a = bf16lo_to_f32(sa[u]), s_b = bf16lo_to_f32(sb[u]);
        a0 = fmaf(s_a, c[0], a0);
        a1 = fmaf(s_a, c[1], a1);
        b0 = fmaf(s_b, c[2], b0);
        b1 = fmaf(s_b, c[3], b1);
    };

    for (int base = 0; base < nG; base += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < nG) {
                compute(u, G0 + base + u);
                if (base + u + U < nG)
                    load(u, G0 + base + u + U);
            }
        }
    }

    m8_store<ARGMAX, PAIRS>(y, a0, a1, b0, b1, M, N, g, t, rowA, rowB, active, ksplit, ks, rbl, rbc,
                            reinterpret_cast<float *>(xs + 8 * cpr), keys);
}

// U = 8 (8 quads in flight, ~160 registers) runs CTAs of at most 12 warps.
// CL4 (no pick, no pairs; a launch with clusters of 4 CTAs): the 4 CTAs of a
// cluster share 4 row blocks, CTA r takes K quarter r of all four (ksplit is
// the split within the CTA), so each CTA stages only its quarter of x; each
// CTA's sums go to the row block's owner (rank = row block within the
// cluster) through distributed shared memory and are added there in rank
// order. At M = 8 the bytes an SM takes in set the x staging time (x is
// 8 K bf16 per CTA: 196 KB at K = 12288).
template <int U, bool ARGMAX, bool PAIRS, bool CL4>
__global__ void __launch_bounds__(U == 8 ? 384 : 512)
w4_decode_m8q_kernel(float *__restrict__ y, const uint16_t *__restrict__ x,
               const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc,
               int M, int N, int K, int ksplit, unsigned long long *__restrict__ keys, int lg)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float recv[CL4 ? 4 * 8 * 16 : 1]; // [sender rank][x-row][row] (CL4)
    if (CL4) // every CTA of the cluster has started before any remote store
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nwarps = blockDim.x >> 5;
    const int rbc = nwarps / ksplit;
    const int ks = warp % ksplit, rbl = warp / ksplit;
    const int crank = CL4 ? (int)cluster_rank() : 0;
    const int nrb = (N + 15) >> 4;
    const int rb = (CL4 ? (int)(blockIdx.x >> 2) * 4 : (int)blockIdx.x * rbc) + rbl;
    const bool active = rb < nrb;
    const int ngroups = K >> 5;
    const int nquads = ngroups >> 2; // 4-group (128-k) units, K % 128 == 0
    const int kst = CL4 ? 4 * ksplit : ksplit, ksi = CL4 ? crank * ksplit + ks : ks;
    const int Q0 = (int)((long long)nquads * ksi / kst);
    const int nQ = (int)((long long)nquads * (ksi + 1) / kst) - Q0;

    const int rowA = rb * 16 + g, rowB = rowA + 8;
    const int rA = min(rowA, N - 1), rB = min(rowB, N - 1);
    // Lane t loads all four words of group 4Q + t (one 128-bit load per row)
    // and the four steps of the quad's groups; a transpose inside the quad then
    // gives lane t word t of each of the four groups, as the mma wants.
    const uint32_t *qA = qw + (size_t)rA * (K >> 3) + 4 * t;
    const uint32_t *qB = qw + (size_t)rB * (K >> 3) + 4 * t;
    const uint16_t *sA = sc + (size_t)rA * (ngroups >> lg);
    const uint16_t *sB = sc + (size_t)rB * (ngroups >> lg);

    uint4 wa[U], wb[U];
    uint2 sa[U], sb[U];
    // The steps of the quad's four 32-code groups 4Q .. 4Q+3 as bf16 pairs
    // (one step per 32 << lg codes).
    auto steps4 = [&](const uint16_t *srow, int Q) -> uint2 {
        if (lg == 0)
            return ldg_nc_u64(srow + 4 * Q);
        if (lg == 1) {
            const uint32_t v = ldg_nc_u32(srow + 2 * Q);
            return make_uint2((v & 0xFFFFu) | (v << 16), (v >> 16) | (v & 0xFFFF0000u));
        }
        const uint32_t v = ldg_nc_u16(srow + ((4 * Q) >> lg));
        return make_uint2(v | (v << 16), v | (v << 16));
    };
    auto load = [&](int u, int Q) {
        wa[u] = ldg_stream_v4(qA + 16 * Q);
        wb[u] = ldg_stream_v4(qB + 16 * Q);
        sa[u] = steps4(sA, Q);
        sb[u] = steps4(sB, Q);
    };

    if (threadIdx.x == 32)
        prefetch_l2_bulk(x, (uint32_t)(M * K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < nQ)
            load(u, Q0 + u);
    pdl_launch_dependents();
    pdl_wait();

    uint4 *xs = reinterpret_cast<uint4 *>(smem); // [8][K/8] permuted chunks
    const int cpr = K >> 3;
    if (CL4) {
        // This CTA's K quarter of each x row (the chunks of its quads), all
        // copies in flight at once, then permuted in place by their owners.
        const int c0 = 16 * (int)((long long)nquads * crank / 4);
        const int nc = 16 * (int)((long long)nquads * (crank + 1) / 4) - c0;
        const uint32_t base = smem_addr(xs);
        for (int i = threadIdx.x; i < M * nc; i += blockDim.x) {
            const int m = i / nc, c = c0 + (i - m * nc);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(base + 16u * (uint32_t)(m * cpr + c)),
                         "l"(x + (size_t)m * K + 8 * c)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        for (int i = threadIdx.x; i < M * nc; i += blockDim.x) {
            const int m = i / nc, c = c0 + (i - m * nc);
            xs[m * cpr + c] = permute_x8(xs[m * cpr + c]);
        }
    } else {
        stage_x_rows_async(xs, x, M, K);
    }
    if (M < 8) // rows M..7 of the B operand are zero
        for (int i = M * cpr + threadIdx.x; i < 8 * cpr; i += blockDim.x)
            xs[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // B column g is x-row g; this lane supplies word t of each group.
    const uint4 *xrow = xs + g * cpr + t;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;

    auto compute = [&](int u, int Q) {
        uint32_t va[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        uint32_t vb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
        quad_transpose4(va, t);
        quad_transpose4(vb, t);
        const uint32_t sw_a[2] = {sa[u].x, sa[u].y}, sw_b[2] = {sb[u].x, sb[u].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int G = 4 * Q + j;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 bx = xrow[4 * G];
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            unpack_word(va[j], a04, a15, a26, a37);
            unpack_word(vb[j], b04, b15, b26, b37);
            mma_16816(c, a04, b04, a15, b15, bx.x, bx.y);
            mma_16816(c, a26, b26, a37, b37, bx.z, bx.w);
            const float s_a = (j & 1) ? bf16hi_to_f32(sw_a[j >> 1]) : bf16lo_to_f32(sw_a[j >> 1]);
            const float s_b = (j & 1) ? bf16hi_to_f32(sw_b[j >> 1]) : bf16lo_to_f32(sw_b[j >> 1]);
            a0 = fmaf(s_a, c[0], a0);
            a1 = fmaf(s_a, c[1], a1);
            b0 = fmaf(s_b, c[2], b0);
            b1 = fmaf(s_b, c[3], b1);
        }
    };

    for (int base = 0; base < nQ; base += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < nQ) {
                compute(u, Q0 + base + u);
                if (base + u + U < nQ)
                    load(u, Q0 + base + u + U);
            }
        }
    }

    if (CL4) {
        // Sums of this CTA's K quarter per (row block, x-row, row), in warp
        // order, stored into the owning CTA's recv[crank]; after the cluster
        // barrier each owner adds the four quarters in rank order.
        float *red = reinterpret_cast<float *>(xs + 8 * cpr); // [rbc][ksplit][8][16]
        red[((rbl * ksplit + ks) * 8 + 2 * t) * 16 + g] = a0;
        red[((rbl * ksplit + ks) * 8 + 2 * t) * 16 + g + 8] = b0;
        red[((rbl * ksplit + ks) * 8 + 2 * t + 1) * 16 + g] = a1;
        red[((rbl * ksplit + ks) * 8 + 2 * t + 1) * 16 + g + 8] = b1;
        __syncthreads();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        const uint32_t rbase = smem_addr(recv);
        for (int i = threadIdx.x; i < rbc * 8 * 16; i += blockDim.x) {
            const int rr = i & 15, mm = (i >> 4) & 7, rl = i >> 7;
            float sum = 0.f;
            for (int k2 = 0; k2 < ksplit; ++k2)
                sum += red[((rl * ksplit + k2) * 8 + mm) * 16 + rr];
            const uint32_t dst = map_rank(rbase + 4u * (uint32_t)((crank * 8 + mm) * 16 + rr), (uint32_t)rl);
            asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(sum) : "memory");
        }
        cluster_sync();
        const int row0 = ((int)(blockIdx.x >> 2) * 4 + crank) * 16;
        for (int i = threadIdx.x; i < 8 * 16; i += blockDim.x) {
            const int rr = i & 15, mm = i >> 4;
            if (mm < M && row0 + rr < N)
                y[(size_t)mm * N + row0 + rr] =
                    ((recv[(0 * 8 + mm) * 16 + rr] + recv[(1 * 8 + mm) * 16 + rr]) + recv[(2 * 8 + mm) * 16 + rr]) +
                    recv[(3 * 8 + mm) * 16 + rr];
        }
        return;
    }
    m8_store<ARGMAX, PAIRS>(y, a0, a1, b0, b1, M, N, g, t, rowA, rowB, active, ksplit, ks, rbl, rbc,
                            reinterpret_cast<float *>(xs + 8 * cpr), keys);
}

// Large N at M <= 8 (the vocabulary projection for up to 8 x-rows): the quad
// kernel's loads and compute, with each warp walking row blocks gw, gw + GW, ...
// of the whole grid as one stream of k-quads (U in flight, the pipeline never
// drains between row blocks), as the M <= 2 large-N form does. A row block's
// outputs (and argmax keys) are stored when its last quad is computed.
// K % 128 == 0, N % 16 == 0, 8-byte-aligned steps; two CTAs of 8 warps per SM.
template <int U, bool ARGMAX, bool PAIRS>
__global__ void __launch_bounds__(256, 2)
w4_decode_m8q_persist_kernel(float *__restrict__ y, const uint16_t *__restrict__ x,
                        const uint32_t *__restrict__ qw, const uint16_t *__restrict__ sc, int M, int N, int K,
                        unsigned long long *__restrict__ keys, int lg, int sc8)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nrb = N >> 4;
    const int ngroups = K >> 5, nq = ngroups >> 2;
    const int GW = gridDim.x * 8, gw = blockIdx.x * 8 + warp;
    const int nmine = nrb > gw ? (nrb - gw + GW - 1) / GW : 0;
    const int Qt = nmine * nq; // k-quads of this warp, row block by row block
    const int sstride = ngroups >> lg;

    // Loader cursor: row A of the warp's current row block (row B is 8 rows on)
    // and the quad within it.
    const uint32_t *lpA = qw + (size_t)(gw * 16 + g) * (K >> 3) + 4 * t;
    const uint16_t *lsA = sc + (size_t)(gw * 16 + g) * sstride;
    const size_t rowB_words = (size_t)8 * (K >> 3), rowB_steps = (size_t)8 * sstride;
    const size_t rb_words = (size_t)GW * 16 * (K >> 3), rb_steps = (size_t)GW * 16 * sstride;
    int lq = 0;

    uint4 wa[U], wb[U];
    uint2 sa[U], sb[U];
    auto steps4 = [&](const uint16_t *srow, int Q) -> uint2 {
        if (!sc8) { // steps not 8-byte aligned: four 16-bit loads
            uint32_t v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = ldg_nc_u16(srow + ((4 * Q + j) >> lg));
            return make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
        }
        if (lg == 0)
            return ldg_nc_u64(srow + 4 * Q);
        if (lg == 1) {
            const uint32_t v = ldg_nc_u32(srow + 2 * Q);
            return make_uint2((v & 0xFFFFu) | (v << 16), (v >> 16) | (v & 0xFFFF0000u));
        }
        const uint32_t v = ldg_nc_u16(srow + ((4 * Q) >> lg));
        return make_uint2(v | (v << 16), v | (v << 16));
    };
    auto load = [&](int u) {
        wa[u] = ldg_stream_v4(lpA + 16 * lq);
        wb[u] = ldg_stream_v4(lpA + rowB_words + 16 * lq);
        sa[u] = steps4(lsA, lq);
        sb[u] = steps4(lsA + rowB_steps, lq);
        if (++lq == nq) {
            lq = 0;
            lpA += rb_words;
            lsA += rb_steps;
        }
    };

    if (threadIdx.x == 32)
        prefetch_l2_bulk(x, (uint32_t)(M * K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < Qt)
            load(u);
    pdl_launch_dependents();
    pdl_wait();

    uint4 *xs = reinterpret_cast<uint4 *>(smem); // [8][K/8] permuted chunks
    const int cpr = K >> 3;
    stage_x_rows_async(xs, x, M, K);
    if (M < 8) // rows M..7 of the B operand are zero
        for (int i = M * cpr + threadIdx.x; i < 8 * cpr; i += blockDim.x)
            xs[i] = make_uint4(0u, 0u, 0u, 0u);
    __shared__ unsigned long long ck[8];
    if (ARGMAX && threadIdx.x < 8)
        ck[threadIdx.x] = 0ull;
    __syncthreads();

    // B column g is x-row g; this lane supplies word t of each group.
    const uint4 *xrow = xs + g * cpr + t;
    const int Mout = PAIRS ? M / 2 : M;
    const int m0 = PAIRS ? t : 2 * t, m1 = 2 * t + 1;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    int cq = 0, crb = 0; // compute cursor: quad and row block (j-th of this warp)

    auto finish = [&]() {
        // Row block gw + crb * GW: lane (g, t) holds y[2t][rowA], y[2t+1][rowA],
        // y[2t][rowB], y[2t+1][rowB] (N % 16 == 0: both rows exist).
        if (PAIRS) {
            a0 += a1;
            b0 += b1;
        }
        const int rowA = (gw + crb * GW) * 16 + g, rowB = rowA + 8;
        const float v[2][2] = {{a0, a1}, {b0, b1}};
        const int rows[2] = {rowA, rowB};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < (PAIRS ? 1 : 2); ++j) {
                const int mm = j ? m1 : m0;
                if (mm < Mout) {
                    y[(size_t)mm * N + rows[h]] = v[h][j];
                    if (ARGMAX)
                        atomicMax(&ck[mm], argmax_key(v[h][j], rows[h]));
                }
            }
        }
        a0 = a1 = b0 = b1 = 0.f;
    };

    auto compute = [&](int u) {
        uint32_t va[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        uint32_t vb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
        quad_transpose4(va, t);
        quad_transpose4(vb, t);
        const uint32_t sw_a[2] = {sa[u].x, sa[u].y}, sw_b[2] = {sb[u].x, sb[u].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int G = 4 * cq + j;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 bx = xrow[4 * G];
            uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
            unpack_word(va[j], a04, a15, a26, a37);
            unpack_word(vb[j], b04, b15, b26, b37);
            mma_16816(c, a04, b04, a15, b15, bx.x, bx.y);
            mma_16816(c, a26, b26, a37, b37, bx.z, bx.w);
            const float s_a = (j & 1) ? bf16hi_to_f32(sw_a[j >> 1]) : bf16lo_to_f32(sw_a[j >> 1]);
            const float s_b = (j & 1) ? bf16hi_to_f32(sw_b[j >> 1]) : bf16lo_to_f32(sw_b[j >> 1]);
            a0 = fmaf(s_a, c[0], a0);
            a1 = fmaf(s_a, c[1], a1);
            b0 = fmaf(s_b, c[2], b0);
            b1 = fmaf(s_b, c[3], b1);
        }
        if (++cq == nq) {
            finish();
            cq = 0;
            ++crb;
        }
    };

    for (int base = 0; base < Qt; base += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < Qt) {
                compute(u);
                if (base + u + U < Qt)
                    load(u);
            }
        }
    }

    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x < Mout)
            keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = ck[threadIdx.x];
    }
}

// ---------------------------------------------------- argmax finalize ----

__global__ void __launch_bounds__(256)
argmax_finalize_kernel(int32_t *__restrict__ argmax, const unsigned long long *__restrict__ keys,
                       int nblocks, const int32_t *__restrict__ forced)
{
    pdl_wait();
    const int m = blockIdx.x;
    if (forced != nullptr) {
        const int32_t f = *forced;
        if (f >= 0) {
            if (threadIdx.x == 0)
                argmax[m] = f;
            return;
        }
    }
    unsigned long long k = 0ull;
    for (int i = threadIdx.x; i < nblocks; i += blockDim.x)
        k = umax64(k, keys[(size_t)m * nblocks + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        k = umax64(k, __shfl_xor_sync(0xFFFFFFFFu, k, o));
    __shared__ unsigned long long wk[8];
    if ((threadIdx.x & 31) == 0)
        wk[threadIdx.x >> 5] = k;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            b = umax64(b, wk[w]);
        argmax[m] = (int32_t)argmax_key_index(b);
    }
}

// ------------------------------------------------------------- launch ----

template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern>
static cudaError_t set_smem(Kern kern, size_t bytes)
{
    if (bytes <= 48 * 1024)
        return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Clusters of 4 CTAs of the M <= 8 quad kernel's cluster form (16 warps,
// shared memory for x at K = 12288) that can be resident at once on the
// current device (clusters must sit in one GPC), cached per device; 0 if the
// query fails.
int m8_cluster_capacity()
{
    static std::atomic<int> cap[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::call_once(once[dev], [dev] {
        int n = 0;
        const size_t smem = (size_t)8 * 12288 * 2 + (size_t)4 * 4 * 8 * 16 * sizeof(float);
        auto ck = w4_decode_m8q_kernel<4, false, false, true>;
        if (cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(4);
            cfg.blockDim = dim3(512);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 4;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, ck, &cfg) != cudaSuccess)
                n = 0;
        }
        cudaGetLastError();
        cap[dev].store(n);
    });
    return cap[dev].load();
}

DecodePlan plan_decode(int M, int N, int K, int num_sms)
{
    DecodePlan p;
    const int nrb = (N + 15) / 16;
    if (M <= 2 && K % (2 * kTileK) == 0 && N % 16 == 0 && nrb >= 2 * num_sms * 16) {
        // At least two row blocks per warp of a full single wave: persistent
        // warps streaming row block after row block.
        p.kernel = 3;
        p.ksplit = 1;
        p.warps = 8;
        p.unroll = 4;
        // Two resident CTAs per SM when both CTAs' x staging fits the SM's shared
        // memory; one otherwise (the walk is the same for any grid).
        p.grid = 2 * decode_smem_bytes(p, M, K) <= kSmemPerSm ? 2 * num_sms : num_sms;
        return p;
    }
    if (M <= 2) {
        // Split K until ~12 warps per SM carry the stream, down to one k-tile
        // per warp, as long as the whole grid is resident at once (a second
        // wave of CTAs costs a full memory round trip). Rows that leave more
        // than 4 k-tiles per warp keep 8 of them in flight (128 registers a
        // thread instead of <= 96).
        const int T = (K + kTileK - 1) / kTileK;
        const int target = num_sms * 12;
        auto make = [&](int ks) {
            DecodePlan q;
            q.kernel = 2;
            q.ksplit = ks;
            q.warps = ks >= 8 ? ks : 8;
            q.unroll = (T + ks - 1) / ks > 4 ? 8 : 4;
            q.grid = (nrb + q.warps / ks - 1) / (q.warps / ks);
            return q;
        };
        auto resident = [&](const DecodePlan &q) {
            const int regs = q.unroll == 8 ? 128 : 96;
            const int per_sm = (65536 / (regs * 32)) / q.warps;
            return (long long)q.grid <= (long long)num_sms * per_sm;
        };
        if (nrb >= 2 * num_sms) {
            // Many row blocks: one CTA per SM with ceil(nrb / SMs) row blocks
            // each, so no SM carries two CTAs' worth of tiles (with 8-warp CTAs
            // 40 of 152 SMs held two and finished ~2-3 us after the rest), and
            // K split as far as 16 warps and the register file allow.
            const int rbc = (nrb + num_sms - 1) / num_sms;
            for (int ks = 16; ks >= 1; ks /= 2) {
                if (ks > T || rbc * ks > 16)
                    continue;
                const int unroll = (T + ks - 1) / ks > 4 ? 8 : 4;
                const int regs = unroll == 8 ? 128 : 96;
                if (rbc * ks * 32 * regs > 65536)
                    continue;
                p.kernel = 2;
                p.ksplit = ks;
                p.warps = rbc * ks;
                p.unroll = unroll;
                p.grid = (nrb + rbc - 1) / rbc;
                return p;
            }
        }
        p = make(1);
        for (int ks = 2; ks <= 16 && ks <= T && (long long)nrb * p.ksplit < target; ks *= 2) {
            const DecodePlan q = make(ks);
            if (!resident(q))
                break;
            p = q;
        }
        return p;
    } else {
        // Same rule as M <= 2: split K (down to 4 groups per warp) until ~12
        // warps per SM carry the stream, while the grid stays one wave.
        const int ngroups = K / 32;
        const int target = num_sms * 12;
        auto make = [&](int ks) {
            DecodePlan q;
            q.kernel = 8;
            q.ksplit = ks;
            q.warps = ks >= 8 ? ks : 8;
            q.unroll = 4;
            q.grid = (nrb + q.warps / ks - 1) / (q.warps / ks);
            return q;
        };
        auto resident = [&](const DecodePlan &q) {
            const int per_sm = (65536 / (96 * 32)) / q.warps;
            return (long long)q.grid <= (long long)num_sms * per_sm;
        };
        if (K % kTileK == 0 && N % 16 == 0 && nrb >= 2 * num_sms * 16) {
            // Vocabulary-sized N: the persistent form, two CTAs of 8 warps per
            // SM, each warp walking at least two row blocks per wave.
            p.kernel = 9;
            p.ksplit = 1;
            p.warps = 8;
            p.unroll = 4;
            p.grid = 2 * decode_smem_bytes(p, M, K) <= kSmemPerSm ? 2 * num_sms : num_sms;
            return p;
        }
        if (nrb >= 2 * num_sms && K % kTileK == 0) {
            // Many row blocks: as for M <= 2, one CTA per SM holding
            // ceil(nrb / SMs) row blocks, K split as far as 16 warps allow;
            // warps with more than 4 quads keep 8 in flight (~160 registers,
            // so at most 12 warps). Measured on GB300 at M = 8: gate|up
            // 24576 x 1536 11.9 -> 9.8 us, 12288 x 1536 7.4 -> 5.6 us.
            const int rbc = (nrb + num_sms - 1) / num_sms;
            const int nq = K / kTileK;
            for (int ks = 16; ks >= 1; ks /= 2) {
                if (ks > nq || rbc * ks > 16)
                    continue;
                const int unroll = (nq + ks - 1) / ks > 4 ? 8 : 4;
                if ((unroll == 8 && rbc * ks > 12) || rbc * ks * 32 * 100 > 65536)
                    continue;
                p.kernel = 8;
                p.ksplit = ks;
                p.warps = rbc * ks;
                p.unroll = unroll;
                p.grid = (nrb + rbc - 1) / rbc;
                return p;
            }
        }
        p = make(1);
        for (int ks = 2; ks <= 16 && ngroups >= 4 * ks && (long long)nrb * p.ksplit < target; ks *= 2) {
            const DecodePlan q = make(ks);
            if (!resident(q))
                break;
            p = q;
        }
        // Long K, one row block per CTA with K over 16 warps (the 1536-row down
        // projections): clusters of 4 CTAs sharing 4 row blocks, each CTA a K
        // quarter of all four (4 warps per row block), so each stages a
        // quarter of x.
        if (p.kernel == 8 && p.ksplit == 16 && p.warps == 16 && K % kTileK == 0 && K >= 4096 && nrb % 4 == 0 &&
            nrb <= num_sms && m8_cluster_capacity() * 4 >= nrb) {
            p.cluster = 4;
            p.ksplit = 4;
            p.grid = nrb;
        }
        return p;
    }
    const int rbc = p.warps / p.ksplit;
    p.grid = (nrb + rbc - 1) / rbc;
    return p;
}

template <int MX, bool ARGMAX, bool PAIRS>
static cudaError_t launch_m2(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                             const uint16_t *sc, int N, int K, unsigned long long *keys, int lg,
                             const int32_t *forced, int hb, cudaStream_t s)
{
    const int Kpad = (K + kTileK - 1) / kTileK * kTileK;
    const int rbc = p.warps / p.ksplit;
    size_t smem = (size_t)MX * Kpad * 2 + 16;
    if (p.ksplit > 1)
        smem += (size_t)rbc * p.ksplit * MX * 16 * sizeof(float);

    const bool sc32 = (K % 64) == 0, full = (K % kTileK) == 0;
    // Groups above 32 take the same kernels with a run-time step shift.
    auto kern = sc32 ? w4_decode_m2_kernel<MX, 4, true, false, ARGMAX, true, PAIRS>
                     : w4_decode_m2_kernel<MX, 4, false, false, ARGMAX, true, PAIRS>;
    if (p.unroll == 8)
        kern = sc32 ? w4_decode_m2_kernel<MX, 8, true, false, ARGMAX, true, PAIRS>
                    : w4_decode_m2_kernel<MX, 8, false, false, ARGMAX, true, PAIRS>;
    if (full)
        kern = p.unroll == 8 ? w4_decode_m2_kernel<MX, 8, true, true, ARGMAX, true, PAIRS>
                             : w4_decode_m2_kernel<MX, 4, true, true, ARGMAX, true, PAIRS>;
    if (lg > 0) { // K % 64 == 0 here
        kern = p.unroll == 8 ? w4_decode_m2_kernel<MX, 8, true, false, ARGMAX, false, PAIRS>
                             : w4_decode_m2_kernel<MX, 4, true, false, ARGMAX, false, PAIRS>;
        if (full)
            kern = p.unroll == 8 ? w4_decode_m2_kernel<MX, 8, true, true, ARGMAX, false, PAIRS>
                                 : w4_decode_m2_kernel<MX, 4, true, true, ARGMAX, false, PAIRS>;
    }
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3(p.grid), dim3(32 * p.warps), smem, s, y, x, qw, sc, N, K, p.ksplit,
                      keys, lg, forced, hb, hb > 0 ? 1.0f / sqrtf((float)hb) : 0.f);
}

template <bool ARGMAX, bool PAIRS>
static cudaError_t launch_m8(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                             const uint16_t *sc, int M, int N, int K, unsigned long long *keys, int lg,
                             cudaStream_t s)
{
    const int rbc = p.warps / p.ksplit;
    size_t smem = (size_t)8 * K * 2;
    if (p.ksplit > 1)
        smem += (size_t)rbc * p.ksplit * 8 * 16 * sizeof(float);
    auto kern = w4_decode_m8_kernel<8, ARGMAX, PAIRS>;
    // 128-bit code loads with a quad transpose when K % 128 == 0 and the steps
    // allow 8-byte loads.
    if (K % kTileK == 0 && (reinterpret_cast<uintptr_t>(sc) & 7) == 0) {
        kern = p.unroll == 8 ? w4_decode_m8q_kernel<8, ARGMAX, PAIRS, false>
                             : w4_decode_m8q_kernel<4, ARGMAX, PAIRS, false>;
        if (!ARGMAX && !PAIRS && p.cluster == 4) {
            auto ck = p.unroll == 8 ? w4_decode_m8q_kernel<8, false, false, true>
                                    : w4_decode_m8q_kernel<4, false, false, true>;
            cudaError_t e = set_smem(ck, smem);
            if (e != cudaSuccess)
                return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(p.grid);
            cfg.blockDim = dim3(32 * p.warps);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = s;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = 4;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            return cudaLaunchKernelEx(&cfg, ck, y, x, qw, sc, M, N, K, p.ksplit, keys, lg);
        }
    }
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3(p.grid), dim3(32 * p.warps), smem, s, y, x, qw, sc, M, N, K,
                      p.ksplit, keys, lg);
}

template <bool ARGMAX, bool PAIRS>
static cudaError_t launch_m8p(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                              const uint16_t *sc, int M, int N, int K, unsigned long long *keys, int lg,
                              cudaStream_t s)
{
    const size_t smem = (size_t)8 * K * 2;
    auto kern = w4_decode_m8q_persist_kernel<4, ARGMAX, PAIRS>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    const int sc8 = (reinterpret_cast<uintptr_t>(sc) & 7) == 0 ? 1 : 0;
    return launch_pdl(kern, dim3(p.grid), dim3(256), smem, s, y, x, qw, sc, M, N, K, keys, lg, sc8);
}

size_t decode_smem_bytes(const DecodePlan &p, int M, int K)
{
    const size_t rbc = (size_t)(p.warps / p.ksplit);
    if (p.kernel == 3)
        return (size_t)M * K * 2 + 16;
    if (p.kernel == 9)
        return (size_t)8 * K * 2;
    if (p.kernel == 2)
        return (size_t)M * ((K + kTileK - 1) / kTileK * kTileK) * 2 + 16 +
               (p.ksplit > 1 ? rbc * p.ksplit * M * 16 * sizeof(float) : 0);
    return (size_t)8 * K * 2 + (p.ksplit > 1 ? rbc * p.ksplit * 8 * 16 * sizeof(float) : 0);
}

template <int MX, bool ARGMAX, bool PAIRS>
static cudaError_t launch_persist(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                                  const uint16_t *sc, int N, int K, unsigned long long *keys, int lg,
                                  const int32_t *forced, int hb, cudaStream_t s)
{
    const size_t smem = (size_t)MX * K * 2 + 16;
    auto kern = lg == 0 ? w4_decode_m2_persist_kernel<MX, 4, 2, ARGMAX, true, PAIRS>
                        : w4_decode_m2_persist_kernel<MX, 4, 2, ARGMAX, false, PAIRS>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, dim3(p.grid), dim3(256), smem, s, y, x, qw, sc, N, K, keys, lg, forced, hb,
                      hb > 0 ? 1.0f / sqrtf((float)hb) : 0.f);
}

template <bool PAIRS>
static cudaError_t dispatch_decode(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                                   const uint16_t *sc, int M, int N, int K, int lg, unsigned long long *keys,
                                   bool am, const int32_t *fo, int hb, cudaStream_t s)
{
    if (p.kernel == 3) {
        if (M == 1 && !PAIRS)
            return am ? launch_persist<1, true, false>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s)
                      : launch_persist<1, false, false>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s);
        return am ? launch_persist<2, true, PAIRS>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s)
                  : launch_persist<2, false, PAIRS>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s);
    }
    if (p.kernel == 2) {
        if (M == 1 && !PAIRS)
            return am ? launch_m2<1, true, false>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s)
                      : launch_m2<1, false, false>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s);
        return am ? launch_m2<2, true, PAIRS>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s)
                  : launch_m2<2, false, PAIRS>(p, y, x, qw, sc, N, K, keys, lg, fo, hb, s);
    }
    if (p.kernel == 9)
        return am ? launch_m8p<true, PAIRS>(p, y, x, qw, sc, M, N, K, keys, lg, s)
                  : launch_m8p<false, PAIRS>(p, y, x, qw, sc, M, N, K, keys, lg, s);
    return am ? launch_m8<true, PAIRS>(p, y, x, qw, sc, M, N, K, keys, lg, s)
              : launch_m8<false, PAIRS>(p, y, x, qw, sc, M, N, K, keys, lg, s);
}

cudaError_t run_decode(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                       const uint16_t *sc, int M, int N, int K, int lg, unsigned long long *keys,
                       int32_t *argmax, cudaStream_t s, bool pairs, const int32_t *forced, int hblock)
{
    const bool am = argmax != nullptr;
    const int32_t *fo = am ? forced : nullptr;
    const int hb = pairs ? hblock : 0;
    cudaError_t e = pairs ? dispatch_decode<true>(p, y, x, qw, sc, M, N, K, lg, keys, am, fo, hb, s)
                          : dispatch_decode<false>(p, y, x, qw, sc, M, N, K, lg, keys, am, fo, hb, s);
    if (e != cudaSuccess || !am)
        return e;
    return run_argmax_finalize(argmax, keys, pairs ? M / 2 : M, p.grid, s, fo);
}

cudaError_t run_argmax_finalize(int32_t *argmax, const unsigned long long *keys, int M, int nblocks,
                                cudaStream_t s, const int32_t *forced)
{
    return launch_pdl(argmax_finalize_kernel, dim3(M), dim3(256), 0, s, argmax, keys, nblocks, forced);
}

} // namespace w4
