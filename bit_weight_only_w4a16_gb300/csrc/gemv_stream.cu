// Decode W4A16 GEMV (M = 1 or 2) with TMA-streamed weights.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
// (decode reads every weight once, straight from the packed 4-bit words, and
// multiplies in registers without a 16-bit copy), the tiling paragraph (a fixed
// tiling per weight shape) and the CUDA-graph paragraph (a decode step is
// hundreds of small kernels replayed as one graph).
//
// Why this shape on GB300. A decode step is a chain of dependent GEMVs of
// 0.25-3 us of HBM time each, a dependent kernel boundary costs ~0.9 us even
// under programmatic dependent launch, and HBM needs ~100 KB in flight per SM.
// So each kernel:
//   1. starts streaming its weight share into a shared-memory ring at once with
//      3-D tensor copies (one op per stage: 64 rows x kus x 256 k of codes, and
//      one for their steps), issued by a producer warp before the kernel waits
//      on the previous one (griddepcontrol.wait); the stream overlaps the
//      previous kernel and the launch gap;
//   2. keeps every SM busy after the wait: rows are split across clusters in
//      whole 64-row groups and K is split across the CTAs of a cluster, whose
//      partial sums are added through distributed shared memory in a fixed
//      rank order (deterministic; no global scratch; no atomics on y);
//   3. stays under half of an SM's shared memory so the next kernel's CTAs can
//      be resident at the same time and stream their weights.
//
// Stages. A stage is 64 rows (4 row blocks) x kus ku of one CTA's K slice; all
// 8 consumer warps read every stage (warp w: row block w & 3, k-tile half
// w >> 2), so stages are consumed and their slots refilled in order and the
// whole ring stays in flight. Codes arrive as [row][ku][128 B] with the
// hardware's 128-byte swizzle (16-byte chunk c of line L lands at chunk
// c ^ (L & 7)); the mma row -> weight row map pairs rows whose lines differ in
// bit 2 of L & 7, so every 8-lane phase of a 128-bit read touches all 32 banks
// once. Steps arrive as [row][ku][8 x bf16] without swizzle.
//
// Inner product: exact (code - 8) bf16 x bf16 m16n8k16 mma with fp32 accumulate.
// Lane (g, t) holds group 4*kt + t of two weight rows; B column 4*m + s carries
// x-row m on group slot s (zero elsewhere), so C[row][4m+s] is the unscaled
// partial of one (row, group, x-row), scaled by its step in fp32.
#include "common.cuh"
#include "internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace w4 {

namespace {

constexpr int kMaxSlots = 16;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kGroupRows = 64;       // rows per stage (4 row blocks of 16)
constexpr int kWaitLimit = 1 << 22;  // polls before a wait is declared failed
constexpr int kDrainLimit = 1 << 10; // polls per wait once a failure was seen
constexpr int kSmemBudget = 110 * 1024;

struct StreamArgs {
    float *y;
    const uint16_t *x;
    unsigned long long *keys; // argmax keys [MX][gridDim.x] or null
    int *err;                 // device error word (bit 0: a wait timed out)
    int N, K;
    int nclusters;   // row-group ranges (one cluster each)
    int kus;         // ku (256-k units) per stage
    int ns;          // ring slots
    int off_steps;   // offset of the steps ring (codes ring at the aligned base)
    int off_x, off_spart, off_rbpart;
    uint32_t perm_lo, perm_hi; // mma row g -> row of the block, 4 bits each (g < 8, g >= 8)
};

struct StreamMaps {
    CUtensorMap codes; // uint32 {32, K/256, N}, box {32, kus, 64}, 128-byte swizzle
    CUtensorMap steps; // uint16 {8, K/256, N},  box {8, kus, 64}
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
                 "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void emit(const StreamArgs &a, int m, int row, float v,
                                     unsigned long long *s_key, bool argmax)
{
    if (row < a.N) {
        a.y[(size_t)m * a.N + row] = v;
        if (argmax)
            atomicMax(&s_key[m], argmax_key(v, (uint32_t)row));
    }
}

template <int MX, bool ARGMAX>
__global__ void __launch_bounds__(kThreads, 2)
gemv_stream_kernel(const StreamArgs a, const __grid_constant__ StreamMaps maps)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full_bar[kMaxSlots];
    __shared__ __align__(8) unsigned long long empty_bar[kMaxSlots];
    __shared__ int s_abort;
    __shared__ unsigned long long s_key[MX];

    // Codes ring on a 1024-byte boundary (the swizzle pattern's period).
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int C = (int)(gridDim.x / a.nclusters);
    const int crank = (C > 1) ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C;
    const int nrg = (a.N + kGroupRows - 1) / kGroupRows;
    const int nku = a.K >> 8;
    const int g0 = (int)((long long)cid * nrg / a.nclusters);
    const int ngc = (int)((long long)(cid + 1) * nrg / a.nclusters) - g0;
    const int ku0 = crank * (nku / C);  // C divides nku
    const int sprg = (nku / C) / a.kus; // stages per row group; kus divides nku / C
    const int nst = ngc * sprg;
    const int code_slot = a.kus * (kGroupRows * 128), step_slot = a.kus * (kGroupRows * 16);

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ns; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), kConsumerWarps);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (ARGMAX && threadIdx.x < MX)
        s_key[threadIdx.x] = 0ull;
    __syncthreads();
    pdl_launch_dependents();

    const uint32_t codes_ring = smem_addr(smem);
    const uint32_t steps_ring = codes_ring + a.off_steps;
    float *spart = reinterpret_cast<float *>(smem + a.off_spart);   // [ngc][8 warps][MX][16]
    float *rbpart = reinterpret_cast<float *>(smem + a.off_rbpart); // [ngc][4][MX][16]

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------- producer warp
        // Weights do not depend on earlier kernels, so no griddepcontrol.wait.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t tx = (uint32_t)(code_slot + step_slot);
            for (int i = 0; i < nst; ++i) {
                const int slot = i % a.ns, use = i / a.ns;
                if (use > 0 && !mbar_wait_bounded(smem_addr(&empty_bar[slot]), (use - 1) & 1,
                                                  s_abort ? kDrainLimit : kWaitLimit)) {
                    s_abort = 1;
                    atomicOr(a.err, 1);
                }
                const int gl = i / sprg, j = i - gl * sprg;
                const int kua = ku0 + j * a.kus;
                const int row0 = (g0 + gl) * kGroupRows;
                const uint32_t bar = smem_addr(&full_bar[slot]);
                mbar_arrive_expect_tx(bar, tx);
                tma_load_3d(codes_ring + slot * code_slot, &maps.codes, 0, kua, row0, bar, pol);
                tma_load_3d(steps_ring + slot * step_slot, &maps.steps, 0, kua, row0, bar, pol);
            }
        }
    } else {
        // -------------------------------------------------- consumer warps
        pdl_wait(); // x may be the previous kernel's output
        uint4 *xs = reinterpret_cast<uint4 *>(smem + a.off_x);
        const int cpr = a.K >> 3;
        for (int i = threadIdx.x; i < MX * cpr; i += kConsumers) {
            const int m = i / cpr, c = i - m * cpr;
            xs[i] = permute_x8(*reinterpret_cast<const uint4 *>(a.x + (size_t)m * a.K + c * 8));
        }
        if (threadIdx.x == 0)
            xs[MX * cpr] = make_uint4(0u, 0u, 0u, 0u);
        named_sync(1, kConsumers);

        const int g = lane >> 2, t = lane & 3;
        const int bm = g >> 2;
        const bool bsel = ((g & 3) == t) && (bm < MX);
        const uint4 *xrow = bsel ? xs + bm * cpr + 4 * t : xs + MX * cpr;
        const int xstep = bsel ? 16 : 0, xi = bsel ? 1 : 0;
        const int rbl = warp & 3;   // row block of the group this warp reads
        const int khalf = warp >> 2; // which half of each stage's k-tiles
        // weight rows (within the 64-row group) of mma rows g and g + 8
        const int ra = rbl * 16 + (int)((a.perm_lo >> (4 * g)) & 15u);
        const int rbr = rbl * 16 + (int)((a.perm_hi >> (4 * g)) & 15u);
        const int la0 = ra * a.kus, lb0 = rbr * a.kus; // first 128-byte line of each row
        const int spoff_a = la0 * 16 + 4 * (t & 1), spoff_b = lb0 * 16 + 4 * (t & 1);

        float accA = 0.f, accB = 0.f;
        for (int i = 0; i < nst; ++i) {
            const int slot = i % a.ns, use = i / a.ns;
            if (!mbar_wait_bounded(smem_addr(&full_bar[slot]), use & 1,
                                   s_abort ? kDrainLimit : kWaitLimit)) {
                if (lane == 0) {
                    s_abort = 1;
                    atomicOr(a.err, 1);
                }
            }
            const int gl = i / sprg, j = i - gl * sprg;
            const int kua = ku0 + j * a.kus;
            const unsigned char *cb = smem + slot * code_slot;
            const unsigned char *sb = smem + a.off_steps + slot * step_slot;
            const uint4 *xb0 = xrow + xstep * (2 * kua);
            for (int kk = 0; kk < a.kus; ++kk) {
                const int kt = khalf * a.kus + kk; // k-tile of the stage (0 .. 2*kus-1)
                const int u = kt >> 1, ch = 4 * (kt & 1) + t;
                const int la = la0 + u, lb = lb0 + u;
                const uint4 wa =
                    *reinterpret_cast<const uint4 *>(cb + la * 128 + ((ch ^ (la & 7)) << 4));
                const uint4 wb =
                    *reinterpret_cast<const uint4 *>(cb + lb * 128 + ((ch ^ (lb & 7)) << 4));
                const uint32_t sa = *reinterpret_cast<const uint32_t *>(sb + spoff_a + u * 16 + 8 * (kt & 1));
                const uint32_t sbv = *reinterpret_cast<const uint32_t *>(sb + spoff_b + u * 16 + 8 * (kt & 1));
                const uint4 *xb = xb0 + xstep * kt;
                const uint32_t aw[4] = {wa.x, wa.y, wa.z, wa.w};
                const uint32_t bw[4] = {wb.x, wb.y, wb.z, wb.w};
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 b = xb[xi * q];
                    uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
                    unpack_word(aw[q], a04, a15, a26, a37);
                    unpack_word(bw[q], b04, b15, b26, b37);
                    mma_16816(c, a04, b04, a15, b15, b.x, b.y);
                    mma_16816(c, a26, b26, a37, b37, b.z, b.w);
                }
                accA = fmaf(bf16lo_to_f32(sa), c[0], accA);
                accA = fmaf(bf16hi_to_f32(sa), c[1], accA);
                accB = fmaf(bf16lo_to_f32(sbv), c[2], accB);
                accB = fmaf(bf16hi_to_f32(sbv), c[3], accB);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty_bar[slot]));
            if (j == sprg - 1) {
                // End of this row group's K slice: park the warp's partials.
                const float pA = accA + __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
                const float pB = accB + __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
                const int m = t >> 1;
                if ((t & 1) == 0 && m < MX) {
                    float *sp = spart + ((gl * kConsumerWarps + warp) * MX + m) * 16;
                    sp[ra - rbl * 16] = pA;
                    sp[rbr - rbl * 16] = pB;
                }
                accA = accB = 0.f;
            }
        }
        named_sync(1, kConsumers);

        // Row block rbl of group gl: its two k-halves (warps rbl, rbl + 4) in order.
        for (int e = threadIdx.x; e < ngc * 4 * MX * 16; e += kConsumers) {
            const int rr = e & 15, m = (e >> 4) % MX, q = e / (16 * MX);
            const int gl = q >> 2, rb = q & 3;
            const float s = spart[((gl * kConsumerWarps + rb) * MX + m) * 16 + rr] +
                            spart[((gl * kConsumerWarps + rb + 4) * MX + m) * 16 + rr];
            if (C == 1)
                emit(a, m, (g0 + gl) * kGroupRows + rb * 16 + rr, s, s_key, ARGMAX);
            else
                rbpart[e] = s;
        }
    }

    if (C > 1) {
        // Add the K slices of the cluster's CTAs in rank order through DSMEM;
        // rank r writes elements [r*E/C, (r+1)*E/C) of the cluster's rows.
        cluster_sync();
        if (warp < kConsumerWarps) {
            const int E = ngc * 4 * MX * 16;
            const int e0 = (int)((long long)crank * E / C), e1 = (int)((long long)(crank + 1) * E / C);
            const uint32_t base = smem_addr(rbpart);
            for (int e = e0 + threadIdx.x; e < e1; e += kConsumers) {
                float s = 0.f;
                for (int c = 0; c < C; ++c)
                    s += ld_cluster_f32(map_rank(base + 4u * e, (uint32_t)c));
                const int rr = e & 15, m = (e >> 4) % MX, q = e / (16 * MX);
                emit(a, m, (g0 + (q >> 2)) * kGroupRows + (q & 3) * 16 + rr, s, s_key, ARGMAX);
            }
        }
        cluster_sync(); // no CTA leaves while another still reads its shared memory
    }

    if (ARGMAX) {
        __syncthreads();
        if (threadIdx.x < MX)
            a.keys[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = s_key[threadIdx.x];
    }
}

// ------------------------------------------------------------ host side ----

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Largest divisor of n that is <= cap.
int divisor_at_most(int n, int cap)
{
    for (int d = cap; d >= 1; --d)
        if (n % d == 0)
            return d;
    return 1;
}

struct Geometry {
    int C = 1, nclusters = 1, kus = 1, ns = 1;
    int off_steps = 0, off_x = 0, off_spart = 0, off_rbpart = 0, smem = 0;
    bool ok = false;
};

// Stage size and slot count for a given split: among kus in {3, 2, 1} that
// divide the CTA's K slice, the one with the most bytes in flight (ties: larger).
Geometry make_geometry(int M, int N, int K, int C, int nclusters)
{
    Geometry G;
    const int nrg = ceil_div(N, kGroupRows), nku = K / 256;
    if (nku % C != 0)
        return G;
    const int nkuc = nku / C;
    const int rgc_max = ceil_div(nrg, nclusters);
    const int x_bytes = M * K * 2 + 16;
    const int spart_bytes = rgc_max * kConsumerWarps * M * 16 * 4;
    const int rbpart_bytes = (C > 1) ? rgc_max * 4 * M * 16 * 4 : 0;
    long long best = -1;
    for (int kus = 3; kus >= 1; --kus) {
        if (nkuc % kus != 0)
            continue;
        const int code_slot = kus * kGroupRows * 128, step_slot = kus * kGroupRows * 16;
        const int max_stages = rgc_max * (nkuc / kus);
        const int fixed = x_bytes + spart_bytes + rbpart_bytes + 1024 + 64;
        int ns = (kSmemBudget - fixed) / (code_slot + step_slot);
        if (ns > kMaxSlots)
            ns = kMaxSlots;
        if (ns > max_stages)
            ns = max_stages;
        if (ns < 1 || (ns < 2 && max_stages > 1))
            continue;
        const long long inflight = (long long)ns * (code_slot + step_slot);
        if (inflight <= best)
            continue;
        best = inflight;
        G.C = C;
        G.nclusters = nclusters;
        G.kus = kus;
        G.ns = ns;
        G.off_steps = ns * code_slot;
        G.off_x = (G.off_steps + ns * step_slot + 15) & ~15;
        G.off_spart = (G.off_x + x_bytes + 15) & ~15;
        G.off_rbpart = (G.off_spart + spart_bytes + 15) & ~15;
        G.smem = G.off_rbpart + rbpart_bytes + 1024; // + alignment slack
        G.ok = true;
    }
    return G;
}

// mma row -> weight row map that keeps 128-bit reads of the swizzled codes
// conflict-free: the two rows read by one 8-lane phase differ in bit 2 of
// (row * kus + u) & 7 for every u < kus (pairs r, r+4 for odd kus; r, r+2 for
// kus = 2 mod 4; r, r+1 for kus = 0 mod 4).
void row_perm(int kus, uint32_t &lo, uint32_t &hi)
{
    int p[16];
    const int d = (kus & 1) ? 4 : ((kus & 3) == 2 ? 2 : 1);
    for (int h = 0; h < 2; ++h) {
        int n = 0;
        for (int r = 0; r < 8 && n < 8; ++r) {
            if ((r / d) % 2 == 0) {
                p[8 * h + n++] = 8 * h + r;
                p[8 * h + n++] = 8 * h + r + d;
            }
        }
    }
    lo = hi = 0;
    for (int g = 0; g < 8; ++g) {
        lo |= (uint32_t)p[g] << (4 * g);
        hi |= (uint32_t)p[8 + g] << (4 * g);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
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

bool encode_maps(StreamMaps &m, const uint32_t *qw, const uint16_t *sc, int N, int K, int kus)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t nku = (cuuint64_t)(K / 256);
    cuuint32_t es[3] = {1, 1, 1};
    {
        cuuint64_t dims[3] = {32, nku, (cuuint64_t)N};
        cuuint64_t strides[2] = {128, (cuuint64_t)K / 2};
        cuuint32_t box[3] = {32, (cuuint32_t)kus, (cuuint32_t)kGroupRows};
        if (enc(&m.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t *>(qw), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t dims[3] = {8, nku, (cuuint64_t)N};
        cuuint64_t strides[2] = {16, (cuuint64_t)K / 16};
        cuuint32_t box[3] = {8, (cuuint32_t)kus, (cuuint32_t)kGroupRows};
        if (enc(&m.steps, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t *>(sc), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

template <int MX, bool ARGMAX>
cudaError_t launch_stream(const Geometry &G, const StreamArgs &a, const StreamMaps &maps,
                          cudaStream_t s)
{
    auto kern = gemv_stream_kernel<MX, ARGMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G.smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G.C * G.nclusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = G.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = G.C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, maps);
}

} // namespace

bool stream_supported(int M, int N, int K, const void *qw, const void *sc)
{
    (void)N;
    return M >= 1 && M <= 2 && K % 256 == 0 && (reinterpret_cast<uintptr_t>(qw) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(sc) & 15) == 0 && tensor_map_encoder() != nullptr;
}

StreamPlan plan_stream(int M, int N, int K, int num_sms)
{
    // Per-shape tiling: the cluster size C (K slices, C | K/256) and the number
    // of clusters (64-row groups split across them) that minimise the largest
    // per-CTA share, one CTA per SM; a share in small tensor copies costs more
    // per byte, weighted by (1 + 1/(2 kus)).
    StreamPlan best;
    const int nrg = ceil_div(N, kGroupRows), nku = K / 256;
    double best_cost = -1.0;
    const int cands[] = {1, 2, 3, 4, 6, 8};
    for (int C : cands) {
        if (nku % C != 0)
            continue;
        int ncl = num_sms / C;
        if (ncl > nrg)
            ncl = nrg;
        if (ncl < 1)
            continue;
        const Geometry G = make_geometry(M, N, K, C, ncl);
        if (!G.ok)
            continue;
        const double cost = (double)ceil_div(nrg, ncl) * (nku / C) * (1.0 + 0.5 / G.kus);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.C = C;
            best.nclusters = ncl;
        }
    }
    best.ok = best_cost >= 0;
    return best;
}

cudaError_t run_stream(const StreamPlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                       const uint16_t *sc, int M, int N, int K, unsigned long long *keys,
                       int32_t *argmax, int *err, cudaStream_t s)
{
    const Geometry G = make_geometry(M, N, K, p.C, p.nclusters);
    if (!G.ok)
        return cudaErrorInvalidConfiguration;
    StreamMaps maps;
    if (!encode_maps(maps, qw, sc, N, K, G.kus))
        return cudaErrorInvalidValue;
    StreamArgs a;
    a.y = y;
    a.x = x;
    a.keys = keys;
    a.err = err;
    a.N = N;
    a.K = K;
    a.nclusters = G.nclusters;
    a.kus = G.kus;
    a.ns = G.ns;
    a.off_steps = G.off_steps;
    a.off_x = G.off_x;
    a.off_spart = G.off_spart;
    a.off_rbpart = G.off_rbpart;
    row_perm(G.kus, a.perm_lo, a.perm_hi);
    const bool am = argmax != nullptr;
    cudaError_t e;
    if (M == 1)
        e = am ? launch_stream<1, true>(G, a, maps, s) : launch_stream<1, false>(G, a, maps, s);
    else
        e = am ? launch_stream<2, true>(G, a, maps, s) : launch_stream<2, false>(G, a, maps, s);
    if (e != cudaSuccess || !am)
        return e;
    return run_argmax_finalize(argmax, keys, M, G.C * G.nclusters, s);
}

} // namespace w4
