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
//      3-D tensor copies (one op per stage for codes, one for steps), issued by
//      a producer warp before the kernel waits
//      on the previous one (griddepcontrol.wait); the stream overlaps the
//      previous kernel and the launch gap;
//   2. keeps every SM busy after the wait: rows are split across clusters in
//      whole 16-row blocks and K is split across the CTAs of a cluster, whose
//      partial sums are added through distributed shared memory in a fixed
//      rank order (deterministic; no global scratch; no atomics on y);
//   3. stays under half of an SM's shared memory so the next kernel's CTAs can
//      be resident at the same time and stream their weights.
//
// Stages. A stage is one 16-row block over the CTA's whole K slice, fetched
// as one 3-D tensor copy of codes ({32 words, ku, 16 rows}: every row a
// contiguous run of K-slice/2 bytes, which is what the copy engine streams
// fastest) and one of steps. All 12 consumer warps read every stage, taking its
// 256-k units in a rotation that balances over consecutive stages, so slots are
// consumed and refilled in order and the whole ring stays in flight; the last
// warp to finish a stage adds the warps' partials in warp order. Codes land
// with the hardware's 128-byte swizzle (16-byte chunk c of line L at chunk
// c ^ (L & 7)); the mma row -> weight row map pairs rows whose lines differ in
// bit 2 of L & 7, so each 8-lane phase of a 128-bit read touches all 32 banks
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
constexpr int kConsumerWarps = 12;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxKu = 16;           // ku per stage (box depth; 4 KB of codes per row)
constexpr int kWaitLimit = 1 << 22;  // polls before a wait is declared failed
constexpr int kDrainLimit = 1 << 10; // polls per wait once a failure was seen
constexpr int kSmemBudget = 110 * 1024;

struct StreamArgs {
    float *y;
    const uint16_t *x;
    unsigned long long *keys; // argmax keys [MX][gridDim.x] or null
    int *err;                 // device error word (bit 0: a wait timed out)
    int N, K;
    int nclusters;   // row-block ranges (one cluster each)
    int ns;          // ring slots
    int off_steps;   // offset of the steps ring (codes ring at the aligned base)
    int off_x, off_red, off_rbpart;
    uint32_t perm_lo, perm_hi; // mma row g -> weight row of the block, 4 bits each
};

struct StreamMaps {
    CUtensorMap codes; // uint32 {32, K/256, N}, box {32, K/256/C, 16}, 128-byte swizzle
    CUtensorMap steps; // uint16 {8, K/256, N},  box {8, K/256/C, 16}
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
    __shared__ int s_count[kMaxSlots];
    __shared__ int s_abort;
    __shared__ unsigned long long s_key[MX];

    // Codes ring on a 1024-byte boundary (the swizzle pattern's period).
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int C = (int)(gridDim.x / a.nclusters);
    const int crank = (C > 1) ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C;
    const int nrb = (a.N + 15) >> 4;
    const int nkuc = (a.K >> 8) / C; // ku of this CTA's K slice (C divides K/256)
    const int ku0 = crank * nkuc;
    const int rb0 = (int)((long long)cid * nrb / a.nclusters);
    const int nst = (int)((long long)(cid + 1) * nrb / a.nclusters) - rb0; // one stage per row block
    const int code_slot = nkuc * 2048, step_slot = nkuc * 256;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ns; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), kConsumerWarps);
            s_count[i] = 0;
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
    float *red = reinterpret_cast<float *>(smem + a.off_red);       // [ns][8 warps][MX][16]
    float *rbpart = reinterpret_cast<float *>(smem + a.off_rbpart); // [nst][MX][16] (C > 1)

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
                const uint32_t bar = smem_addr(&full_bar[slot]);
                mbar_arrive_expect_tx(bar, tx);
                tma_load_3d(codes_ring + slot * code_slot, &maps.codes, 0, ku0, (rb0 + i) * 16, bar, pol);
                tma_load_3d(steps_ring + slot * step_slot, &maps.steps, 0, ku0, (rb0 + i) * 16, bar, pol);
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
        const uint4 *xrow = (bsel ? xs + bm * cpr + 4 * t : xs + MX * cpr);
        const int xstep = bsel ? 16 : 0, xi = bsel ? 1 : 0;
        const uint4 *xb0 = xrow + xstep * (2 * ku0);
        const int ra = (int)((a.perm_lo >> (4 * g)) & 15u);  // weight row of mma row g
        const int rbr = (int)((a.perm_hi >> (4 * g)) & 15u); // weight row of mma row g + 8
        const int la0 = ra * nkuc, lb0 = rbr * nkuc;         // first 128-byte line of each row

        for (int i = 0; i < nst; ++i) {
            const int slot = i % a.ns, use = i / a.ns;
            if (!mbar_wait_bounded(smem_addr(&full_bar[slot]), use & 1,
                                   s_abort ? kDrainLimit : kWaitLimit)) {
                if (lane == 0) {
                    s_abort = 1;
                    atomicOr(a.err, 1);
                }
            }
            const uint32_t cb = codes_ring + slot * code_slot;
            const uint32_t sbase = steps_ring + slot * step_slot;
            float accA = 0.f, accB = 0.f;
            // 256-k units u = first, first + 8, ...; the rotation balances the
            // warps over consecutive stages.
            const int first = (int)((((unsigned)warp + (unsigned)kConsumerWarps * 4096u) - (unsigned)((i * nkuc) % kConsumerWarps)) % (unsigned)kConsumerWarps);
            for (int u = first; u < nkuc; u += kConsumerWarps) {
                const int la = la0 + u, lb = lb0 + u;
                // 16-byte chunk t of k-tile 0 and chunk 4 + t of k-tile 1, swizzled
                const uint32_t qa0 = cb + la * 128 + ((t ^ (la & 7)) << 4);
                const uint32_t qb0 = cb + lb * 128 + ((t ^ (lb & 7)) << 4);
                const uint4 wa0 = lds128(qa0), wa1 = lds128(qa0 ^ 64u);
                const uint4 wb0 = lds128(qb0), wb1 = lds128(qb0 ^ 64u);
                const uint32_t pa = sbase + la * 16 + 4 * (t & 1);
                const uint32_t pb = sbase + lb * 16 + 4 * (t & 1);
                const uint32_t sa0 = lds32(pa), sa1 = lds32(pa + 8);
                const uint32_t sb0 = lds32(pb), sb1 = lds32(pb + 8);
                const uint4 *xb = xb0 + xstep * (2 * u);
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t a0w[4] = {wa0.x, wa0.y, wa0.z, wa0.w}, b0w[4] = {wb0.x, wb0.y, wb0.z, wb0.w};
                const uint32_t a1w[4] = {wa1.x, wa1.y, wa1.z, wa1.w}, b1w[4] = {wb1.x, wb1.y, wb1.z, wb1.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 x0 = xb[xi * q], x1 = xb[xstep + xi * q];
                    uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
                    unpack_word(a0w[q], a04, a15, a26, a37);
                    unpack_word(b0w[q], b04, b15, b26, b37);
                    mma_16816(c0, a04, b04, a15, b15, x0.x, x0.y);
                    mma_16816(c0, a26, b26, a37, b37, x0.z, x0.w);
                    unpack_word(a1w[q], a04, a15, a26, a37);
                    unpack_word(b1w[q], b04, b15, b26, b37);
                    mma_16816(c1, a04, b04, a15, b15, x1.x, x1.y);
                    mma_16816(c1, a26, b26, a37, b37, x1.z, x1.w);
                }
                accA = fmaf(bf16lo_to_f32(sa0), c0[0], accA);
                accA = fmaf(bf16hi_to_f32(sa0), c0[1], accA);
                accB = fmaf(bf16lo_to_f32(sb0), c0[2], accB);
                accB = fmaf(bf16hi_to_f32(sb0), c0[3], accB);
                accA = fmaf(bf16lo_to_f32(sa1), c1[0], accA);
                accA = fmaf(bf16hi_to_f32(sa1), c1[1], accA);
                accB = fmaf(bf16lo_to_f32(sb1), c1[2], accB);
                accB = fmaf(bf16hi_to_f32(sb1), c1[3], accB);
            }
            // This warp's partial of the row block -> red[slot][warp].
            accA += __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
            accB += __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
            const int m = t >> 1;
            float *rs = red + slot * (kConsumerWarps * MX * 16);
            if ((t & 1) == 0 && m < MX) {
                rs[(warp * MX + m) * 16 + ra] = accA;
                rs[(warp * MX + m) * 16 + rbr] = accB;
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = (atomicAdd(&s_count[slot], 1) == kConsumerWarps - 1);
                if (last)
                    __threadfence_block();
            }
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            if (last) {
                // Sum the warps' partials in warp order; reset the counter
                // before the slot is released.
                if (lane < MX * 16) {
                    float s = 0.f;
                    for (int w = 0; w < kConsumerWarps; ++w)
                        s += rs[w * MX * 16 + lane];
                    const int mm = lane >> 4, rr = lane & 15;
                    if (C == 1)
                        emit(a, mm, (rb0 + i) * 16 + rr, s, s_key, ARGMAX);
                    else
                        rbpart[i * MX * 16 + lane] = s;
                }
                if (lane == 0)
                    s_count[slot] = 0;
                __syncwarp();
            }
            if (lane == 0)
                mbar_arrive(smem_addr(&empty_bar[slot]));
        }
    }

    if (C > 1) {
        // Add the K slices of the cluster's CTAs in rank order through DSMEM;
        // rank r writes elements [r*E/C, (r+1)*E/C) of the cluster's rows.
        cluster_sync();
        if (warp < kConsumerWarps) {
            const int E = nst * MX * 16;
            const int e0 = (int)((long long)crank * E / C), e1 = (int)((long long)(crank + 1) * E / C);
            const uint32_t base = smem_addr(rbpart);
            for (int e = e0 + threadIdx.x; e < e1; e += kConsumers) {
                float s = 0.f;
                for (int c = 0; c < C; ++c)
                    s += ld_cluster_f32(map_rank(base + 4u * e, (uint32_t)c));
                const int rr = e & 15, m = (e >> 4) % MX, q = e / (16 * MX);
                emit(a, m, (rb0 + q) * 16 + rr, s, s_key, ARGMAX);
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

struct Geometry {
    int C = 1, nclusters = 1, ns = 1;
    int off_steps = 0, off_x = 0, off_red = 0, off_rbpart = 0, smem = 0;
    bool ok = false;
};

// Ring for a given split: as many whole-stage slots as the budget allows.
Geometry make_geometry(int M, int N, int K, int C, int nclusters)
{
    Geometry G;
    const int nrb = ceil_div(N, 16), nku = K / 256;
    if (nku % C != 0 || nku / C > kMaxKu)
        return G;
    const int nkuc = nku / C;
    const int max_stages = ceil_div(nrb, nclusters);
    const int code_slot = nkuc * 2048, step_slot = nkuc * 256;
    const int red_slot = kConsumerWarps * M * 16 * 4;
    const int x_bytes = M * K * 2 + 16;
    const int rbpart_bytes = (C > 1) ? max_stages * M * 16 * 4 : 0;
    const int fixed = x_bytes + rbpart_bytes + 1024 + 64;
    int ns = (kSmemBudget - fixed) / (code_slot + step_slot + red_slot);
    if (ns > kMaxSlots)
        ns = kMaxSlots;
    if (ns > max_stages)
        ns = max_stages;
    if (ns < 1 || (ns < 2 && max_stages > 1))
        return G;
    G.C = C;
    G.nclusters = nclusters;
    G.ns = ns;
    G.off_steps = ns * code_slot;
    G.off_x = (G.off_steps + ns * step_slot + 15) & ~15;
    G.off_red = (G.off_x + x_bytes + 15) & ~15;
    G.off_rbpart = (G.off_red + ns * red_slot + 15) & ~15;
    G.smem = G.off_rbpart + rbpart_bytes + 1024; // + alignment slack
    G.ok = true;
    return G;
}

// mma row -> weight row map that keeps 128-bit reads of the swizzled codes
// conflict-free: the two rows read by one 8-lane phase differ in bit 2 of
// (row * kus + u) & 7 for every u < kus (pairs r, r+4 for odd kus; r, r+2 for
// kus = 2 mod 4; r, r+1 for kus = 4 mod 8; kus = 0 mod 8 has no such pairing
// and reads with two-way conflicts).
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
        cuuint32_t box[3] = {32, (cuuint32_t)kus, 16};
        if (enc(&m.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t *>(qw), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t dims[3] = {8, nku, (cuuint64_t)N};
        cuuint64_t strides[2] = {16, (cuuint64_t)K / 16};
        cuuint32_t box[3] = {8, (cuuint32_t)kus, 16};
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
    // Per-shape tiling: cluster size C (K slices, C | K/256, at most 16 ku per
    // slice) and the number of clusters (16-row blocks split across them), one
    // CTA per SM. Modelled time of the busiest CTA: its stages, each costing the
    // larger of the copy engine's per-row cost (~40 cycles per row segment) and
    // the segment's bytes at ~24 B/cycle.
    StreamPlan best;
    const int nrb = ceil_div(N, 16), nku = K / 256;
    double best_cost = -1.0;
    const int cands[] = {1, 2, 3, 4, 6, 8};
    for (int C : cands) {
        if (nku % C != 0 || nku / C > kMaxKu)
            continue;
        int ncl = num_sms / C;
        if (ncl > nrb)
            ncl = nrb;
        if (ncl < 1)
            continue;
        const Geometry G = make_geometry(M, N, K, C, ncl);
        if (!G.ok)
            continue;
        const double seg = (double)(nku / C) * 128.0;
        const double per_stage = 16.0 * (seg / 24.0 > 40.0 ? seg / 24.0 : 40.0);
        const double cost = (double)ceil_div(nrb, ncl) * per_stage;
        if (best_cost < 0 || cost < best_cost * 0.999) {
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
    const int nkuc = (K / 256) / G.C;
    StreamMaps maps;
    if (!encode_maps(maps, qw, sc, N, K, nkuc))
        return cudaErrorInvalidValue;
    StreamArgs a;
    a.y = y;
    a.x = x;
    a.keys = keys;
    a.err = err;
    a.N = N;
    a.K = K;
    a.nclusters = G.nclusters;
    a.ns = G.ns;
    a.off_steps = G.off_steps;
    a.off_x = G.off_x;
    a.off_red = G.off_red;
    a.off_rbpart = G.off_rbpart;
    row_perm(nkuc, a.perm_lo, a.perm_hi);
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
