// Decode-form W4A16 GEMV for one activation row (M = 1).
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
// (decode multiplies one vector by every weight matrix: the kernel reads the
// packed 4-bit words, unpacks them in registers and multiplies, never writing a
// 16-bit copy), the tiling paragraph (each weight shape gets its own fixed
// tiling) and the CUDA-graph paragraph (a decode step is a long chain of small
// dependent kernels).
//
// GB300 design. Inside a graph-replayed decode step every call waits for the
// previous one (programmatic dependent launch), so a call's time is: the wait
// release, the x round trip after it, the post-x work of the busiest SM and the
// reduction. Measured per CTA with the SM clock on GB300 (the 35-layer sweep):
// release ~0.75 us, x ~0.75-1.0 us, reduction + store ~0.4 us; the compute is
// issue-bound (~170 warp instructions per 16 x 128 tile). Hence:
//   * a CTA owns R whole 16-row blocks; warp w owns K sub-slice w mod S of
//     its row blocks w / S,
//     w / S + W / S, ... and streams their tiles with running pointers;
//   * after the wait the x loads are issued first and the first preloaded tile
//     is unpacked while they are in flight, so that unpack hides in the x round
//     trip;
//   * B fragments of x are read with compile-time offsets (lanes that feed a
//     zero column read a zero region placed on other banks);
//   * the sub-slices' partials are added in a fixed order through shared
//     memory (deterministic, no atomics on y).
//
// Inner product as in the other decode kernels: lane (g, t) holds one 32-code
// group (16 B) of rows g and g + 8; B column s carries x restricted to group
// slot s (columns 4..7 are zero at M = 1), so C[row][s] is the unscaled partial
// of one (row, group), scaled by its bf16 step in fp32.
#include "common.cuh"
#include "internal.h"

namespace w4 {

namespace {

constexpr int kTile = 128; // k per tile: 4 groups of 32

struct M1Args {
    float *y;
    const uint16_t *x;
    const uint32_t *qw;
    const uint16_t *sc;
    int N, K, lg;
    int R; // 16-row blocks per CTA
    int S; // K sub-slices (warps sharing a row block): sub-slice s is tiles [T*s/S, T*(s+1)/S)
};

// Four words (codes of rows g and g + 8) unpacked to the A operands of two
// m16n8k16 mmas: A[0..3] for codes (0,4)/(1,5), A[4..7] for (2,6)/(3,7).
__device__ __forceinline__ void unpack_words(uint32_t wa, uint32_t wb, uint32_t (&A)[8])
{
    asm("{\n"
        ".reg .b32 t, m, o, k;\n"
        "mov.b32 m, 0x000F000F;\n"
        "mov.b32 o, 0x43004300;\n"
        "mov.b32 k, 0x43084308;\n"
        "lop3.b32 %0, %8, m, o, 0xEA;\n"
        "lop3.b32 %1, %9, m, o, 0xEA;\n"
        "shr.u32 t, %8, 4;\n lop3.b32 %2, t, m, o, 0xEA;\n"
        "shr.u32 t, %9, 4;\n lop3.b32 %3, t, m, o, 0xEA;\n"
        "shr.u32 t, %8, 8;\n lop3.b32 %4, t, m, o, 0xEA;\n"
        "shr.u32 t, %9, 8;\n lop3.b32 %5, t, m, o, 0xEA;\n"
        "shr.u32 t, %8, 12;\n lop3.b32 %6, t, m, o, 0xEA;\n"
        "shr.u32 t, %9, 12;\n lop3.b32 %7, t, m, o, 0xEA;\n"
        "sub.rn.bf16x2 %0, %0, k;\n sub.rn.bf16x2 %1, %1, k;\n"
        "sub.rn.bf16x2 %2, %2, k;\n sub.rn.bf16x2 %3, %3, k;\n"
        "sub.rn.bf16x2 %4, %4, k;\n sub.rn.bf16x2 %5, %5, k;\n"
        "sub.rn.bf16x2 %6, %6, k;\n sub.rn.bf16x2 %7, %7, k;\n"
        "}\n"
        : "=r"(A[0]), "=r"(A[1]), "=r"(A[2]), "=r"(A[3]), "=r"(A[4]), "=r"(A[5]), "=r"(A[6]), "=r"(A[7])
        : "r"(wa), "r"(wb));
}

__device__ __forceinline__ void mma_pair(float (&c)[4], float (&d)[4], const uint32_t (&A)[8], uint4 b)
{
    mma_16816(c, A[0], A[1], A[2], A[3], b.x, b.y);
    mma_16816(d, A[4], A[5], A[6], A[7], b.z, b.w);
}

// U: tiles in flight per warp; the first one is unpacked while x travels.
template <bool G32, int U>
__global__ void __launch_bounds__(512, 1) w4_decode_m1_kernel(const M1Args a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nrb = a.N >> 4;
    const int rb0 = blockIdx.x * a.R;
    const int Rn = min(a.R, nrb - rb0);
    const int S = a.S, Tc = a.K / kTile;
    const int s = warp % S;              // this warp's sub-slice: tiles [ts0, ts0 + Ts)
    const int ts0 = Tc * s / S, Ts = Tc * (s + 1) / S - ts0;
    const int rf = warp / S, rs = W / S; // row blocks rf, rf + rs, ... (local)
    const int nsub = rf < Rn && Ts > 0 ? (Rn - rf + rs - 1) / rs : 0;
    const int Q = nsub * Ts; // tiles of this warp
    const int kw = a.K >> 3; // words per row

    // Shared memory: x (Tc*16 chunks, permuted), zero region (4 chunks, on
    // other banks than the x chunks read in the same phase), partials [Rn][S][16].
    uint4 *xs = reinterpret_cast<uint4 *>(smem);
    const int nchunk = Tc * 16;
    uint4 *zs = xs + nchunk + 2;
    float *red = reinterpret_cast<float *>(zs + 6);

    // Loader cursor: row A of the current row block at the current tile; row B
    // is 8 rows (K words) on. Steps: one per 32 << lg codes.
    const int sstride = (a.K >> 5) >> a.lg;
    const size_t row0 = (size_t)(rb0 + rf) * 16 + g;
    const uint32_t *lp = a.qw + row0 * kw + (size_t)ts0 * 16 + 4 * t;
    const uint16_t *ls = a.sc + row0 * sstride;
    const int lj0 = 4 * ts0 + 2 * (t & 1);
    int lj = lj0, ll = 0;
    const size_t jump_w = (size_t)rs * 16 * kw - (size_t)Ts * 16;
    const size_t jump_s = (size_t)rs * 16 * sstride;
    const size_t rowB_s = (size_t)8 * sstride;

    uint4 wa[U], wb[U];
    uint32_t sa[U], sb[U];
    auto load = [&](int u) {
        wa[u] = ldg_stream_v4(lp);
        wb[u] = ldg_stream_v4(lp + a.K);
        if (G32) {
            sa[u] = ldg_nc_u32(ls + lj);
            sb[u] = ldg_nc_u32(ls + rowB_s + lj);
        } else {
            sa[u] = ldg_nc_u16(ls + (lj >> a.lg));
            sb[u] = ldg_nc_u16(ls + rowB_s + (lj >> a.lg));
        }
        lp += 16;
        lj += 4;
        if (++ll == Ts) {
            ll = 0;
            lp += jump_w;
            ls += jump_s;
            lj = lj0;
        }
    };

    if (threadIdx.x == 32)
        prefetch_l2_bulk(a.x, (uint32_t)(a.K * 2));
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < Q)
            load(u);
    pdl_launch_dependents();
    pdl_wait();

    // x loads first (all of a thread's chunks in flight), then the first tile's
    // unpack while they travel, then the permuted x into shared memory.
    constexpr int kXL = 4;
    uint4 xv[kXL];
    const uint16_t *xg = a.x;
#pragma unroll
    for (int j = 0; j < kXL; ++j) {
        const int i = threadIdx.x + j * blockDim.x;
        xv[j] = i < nchunk ? *reinterpret_cast<const uint4 *>(xg + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t A0[4][8];
    if (Q > 0) {
        const uint32_t wa0[4] = {wa[0].x, wa[0].y, wa[0].z, wa[0].w};
        const uint32_t wb0[4] = {wb[0].x, wb[0].y, wb[0].z, wb[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            unpack_words(wa0[i], wb0[i], A0[i]);
    }
#pragma unroll
    for (int j = 0; j < kXL; ++j) {
        const int i = threadIdx.x + j * blockDim.x;
        if (i < nchunk)
            xs[i] = permute_x8(xv[j]);
    }
    // The rare slice longer than kXL chunks per thread.
    for (int i = threadIdx.x + kXL * blockDim.x; i < nchunk; i += blockDim.x)
        xs[i] = permute_x8(*reinterpret_cast<const uint4 *>(xg + 8 * i));
    if (threadIdx.x < 4)
        zs[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    // B column g = group slot g (g < 4) lives on lane t == g; the other lanes
    // read the zero region (a fixed address per load: broadcast).
    const bool bsel = g < 4 && t == g;
    const uint4 *xbase = bsel ? xs + (size_t)ts0 * 16 + 4 * t : zs;
    const int xstep = bsel ? 16 : 0;
    const uint4 *xc = xbase;

    float accA = 0.f, accB = 0.f;
    int cl = 0, cj = 0; // compute cursor: tile in sub-unit, sub-unit index
    auto finish_tile = [&]() {
        xc += xstep;
        if (++cl == Ts) {
            // Lanes t and t ^ 1 hold group slots (0, 1) and (2, 3) of the row.
            const float vA = accA + __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
            const float vB = accB + __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
            if (t == 0) {
                float *r = red + ((rf + cj * rs) * S + s) * 16;
                r[g] = vA;
                r[g + 8] = vB;
            }
            accA = accB = 0.f;
            cl = 0;
            ++cj;
            xc = xbase;
        }
    };
    auto scale = [&](int u, const float (&c)[4], const float (&d)[4]) {
        if (G32) {
            accA = fmaf(bf16lo_to_f32(sa[u]), c[0] + d[0], accA);
            accA = fmaf(bf16hi_to_f32(sa[u]), c[1] + d[1], accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), c[2] + d[2], accB);
            accB = fmaf(bf16hi_to_f32(sb[u]), c[3] + d[3], accB);
        } else { // both groups of the lane's pair share one step
            accA = fmaf(bf16lo_to_f32(sa[u]), (c[0] + d[0]) + (c[1] + d[1]), accA);
            accB = fmaf(bf16lo_to_f32(sb[u]), (c[2] + d[2]) + (c[3] + d[3]), accB);
        }
    };

    if (Q > 0) { // tile 0: already unpacked
        float c[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mma_pair(c, d, A0[i], xc[i]);
        scale(0, c, d);
        finish_tile();
        if (U < Q)
            load(0);
    }
    for (int base = 0; base < Q; base += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u;
            if ((u == 0 && base == 0) || i >= Q)
                continue;
            float c[4] = {0.f, 0.f, 0.f, 0.f}, d[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t aw[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
            const uint32_t bw[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 b = xc[k];
                unpack_mma2(c, d, aw[k], bw[k], b.x, b.y, b.z, b.w);
            }
            scale(u, c, d);
            finish_tile();
            if (i + U < Q)
                load(u);
        }
    }
    __syncthreads();

    // The sub-slices of each row block, added in order.
    const int nout = Rn * 16;
    float *yb = a.y + (size_t)rb0 * 16;
    for (int o = threadIdx.x; o < nout; o += blockDim.x) {
        const float *r = red + (o >> 4) * S * 16 + (o & 15);
        float v = r[0];
        for (int k = 1; k < S; ++k)
            v += r[16 * k];
        yb[o] = v;
    }
}

size_t m1_smem_bytes(const M1Plan &p)
{
    return (size_t)(p.T * 16 + 8) * 16 + (size_t)p.R * p.S * 16 * 4;
}

} // namespace

M1Plan plan_decode_m1(int M, int N, int K, int num_sms)
{
    // Chosen from measurements on GB300 in the graph-replayed decode sweep:
    //  * each CTA owns whole rows. Splitting K across the CTAs of a cluster
    //    (sizes 3 and up, ~144 SMs for the 1536-row projections) made every
    //    such call slower (1536 x 12288 5.5 -> 7.2 us, 2560 x 1536 2.5 -> 3.5
    //    us): a cluster waits for several SMs of one GPC to free up under the
    //    previous call, and adds two cluster barriers;
    //  * the smallest CTA that keeps each warp at <= 4 tiles wins: 8 warps (two
    //    CTAs can share an SM) took 2560 x 1536 from 2.47 to 2.24 us and
    //    1536 x 2048 from 2.41 to 2.15 us against the register-preload kernel;
    //  * longer warp streams stay with the register-preload kernel, which keeps
    //    8 tiles a warp in flight without this form's extra cursor state
    //    (24576 x 1536 6.9 vs 7.6 us, 1536 x 12288 5.5 vs 5.6-5.9 us).
    M1Plan best;
    if (M != 1 || K % kTile != 0 || N % 16 != 0 || num_sms < 1)
        return best;
    const int T = K / kTile, nrb = N / 16;
    if (nrb >= 2 * num_sms * 16) // vocabulary-sized: the persistent form streams it better
        return best;
    const int Ws[] = {8, 12, 16};
    for (int W : Ws) {
        const int per_sm = W <= 8 ? 2 : 1; // CTAs an SM holds (<= 128 registers a thread)
        const int R = (nrb + per_sm * num_sms - 1) / (per_sm * num_sms);
        const int grid = (nrb + R - 1) / R;
        const int load = (grid + num_sms - 1) / num_sms; // CTAs on the busiest SM
        double best_cost = 1e30;
        M1Plan cand;
        int cand_wmax = 0;
        for (int S = 1; S <= W && S <= T; ++S) {
            if (W % S != 0)
                continue;
            const int rs = W / S;
            // Tiles per SM sub-partition (warp w on partition w % 4) and per warp.
            int part[4] = {0, 0, 0, 0}, wmax = 0, nsub0 = 0;
            for (int w = 0; w < W; ++w) {
                const int sw = w % S, rf = w / S;
                const int ts = T * (sw + 1) / S - T * sw / S;
                const int nsub = rf < R && ts > 0 ? (R - rf + rs - 1) / rs : 0;
                part[w & 3] += nsub * ts;
                wmax = nsub * ts > wmax ? nsub * ts : wmax;
                nsub0 = nsub > nsub0 ? nsub : nsub0;
            }
            int pmax = 0;
            for (int k = 0; k < 4; ++k)
                pmax = part[k] > pmax ? part[k] : pmax;
            // Issue-bound tiles of the busiest partition (times the CTAs that
            // share the SM), the longest warp chain, and the partial flushes.
            const double cost = load * pmax + 0.5 * wmax + (S > 1 ? 0.25 : 0.0) + 0.25 * nsub0;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                cand.ok = true;
                cand.R = R;
                cand.S = S;
                cand.T = T;
                cand.warps = W;
                cand.grid = grid;
                cand_wmax = wmax;
            }
        }
        if (cand.ok && cand_wmax <= 4 && m1_smem_bytes(cand) <= 200 * 1024)
            return cand;
    }
    return best;
}

template <bool G32, int U>
static cudaError_t launch_m1(const M1Plan &p, const M1Args &a, cudaStream_t s)
{
    auto kern = w4_decode_m1_kernel<G32, U>;
    const size_t smem = m1_smem_bytes(p);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(32 * p.warps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t run_decode_m1(const M1Plan &p, float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc,
                          int N, int K, int lg, cudaStream_t s)
{
    if (!p.ok)
        return cudaErrorInvalidConfiguration;
    M1Args a;
    a.y = y;
    a.x = x;
    a.qw = qw;
    a.sc = sc;
    a.N = N;
    a.K = K;
    a.lg = lg;
    a.R = p.R;
    a.S = p.S;
    return lg == 0 ? launch_m1<true, 4>(p, a, s) : launch_m1<false, 4>(p, a, s);
}

} // namespace w4
