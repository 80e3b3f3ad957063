// Decode W4A16 GEMV (M = 1 or 2) with bulk-copy weight streaming.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
// (decode reads every weight once, straight from the packed 4-bit words, and
// multiplies in registers without a 16-bit copy), the tiling paragraph (a fixed
// tiling per weight shape) and the CUDA-graph paragraph (a decode step is
// hundreds of small kernels replayed as one graph).
//
// Why this shape on GB300. A decode step is a chain of dependent GEMVs of
// 0.25-3 us of HBM time each, and a dependent kernel boundary costs ~0.9 us even
// under programmatic dependent launch. So each kernel:
//   1. starts streaming its whole weight share into shared memory at once
//      (1-D bulk copies issued by one producer warp, completion on mbarriers),
//      before waiting on the previous kernel (griddepcontrol.wait), so the
//      stream overlaps the previous kernel and the launch gap;
//   2. keeps every SM busy after the wait: rows are split across clusters in
//      whole 16-row blocks and K is split across the CTAs of a cluster, whose
//      partial sums are added through distributed shared memory in a fixed
//      rank order (deterministic, no global scratch, no atomics on y);
//   3. stays under half of an SM's shared memory so the next kernel's CTAs can
//      be resident at the same time and stream their weights.
//
// Work unit ("ku"): 16 rows x 256 k = 2 KB of codes + 256 B of steps. A stage
// is up to `kus` consecutive ku of one row block, copied row by row into a
// ring slot with a row pitch of 64 mod 128 bytes (conflict-free 128-bit reads).
// Stage i belongs to consumer warp i % 8 and to one of that warp's own `dpw`
// slots, so every slot's mbarrier phases are waited on in order by one warp
// (a parity wait cannot tell phase u from phase u - 2).
//
// Inner product: the exact (code - 8) bf16 x bf16 m16n8k16 mma scheme of the
// register-streaming decode kernel: lane (g, t) holds group 4*kt + t of rows g
// and g+8; B column 4*m + s carries x-row m on group slot s; the group step is
// applied in fp32 per (row, group).
#include "common.cuh"
#include "internal.h"

namespace w4 {

namespace {

constexpr int kMaxSlots = 16;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kWaitLimit = 1 << 22;  // polls before a wait is declared failed
constexpr int kDrainLimit = 1 << 10; // polls per wait once a failure was seen
constexpr int kSmemBudget = 110 * 1024;

struct StreamArgs {
    float *y;
    const uint16_t *x;
    const uint32_t *qw;
    const uint16_t *sc;
    unsigned long long *keys; // argmax keys [MX][gridDim.x] or null
    int *err;                 // device error word (bit 0: a wait timed out)
    int N, K;
    int nclusters;  // row-block groups (one cluster each)
    int kus;        // max ku per stage
    int ns;         // ring slots in use (<= kMaxSlots)
    int dpw;        // ring slots per consumer warp (1 or 2)
    int slot_bytes; // bytes per ring slot
    int pq, ps;     // smem row pitches of codes and steps inside a slot
    int off_x, off_spart, off_rbpart;
};

template <int MX>
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
gemv_stream_kernel(const StreamArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long full_bar[kMaxSlots];
    __shared__ __align__(8) unsigned long long empty_bar[kMaxSlots];
    __shared__ int s_abort;
    __shared__ unsigned long long s_key[MX];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int C = (int)(gridDim.x / a.nclusters);
    const int crank = (C > 1) ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C;
    const int nrb = (a.N + 15) >> 4;
    const int nku = a.K >> 8;
    const int rb0 = (int)((long long)cid * nrb / a.nclusters);
    const int nrbc = (int)((long long)(cid + 1) * nrb / a.nclusters) - rb0;
    const int ku0 = (int)((long long)crank * nku / C);
    const int nkuc = (int)((long long)(crank + 1) * nku / C) - ku0;
    const int sprb = (nkuc + a.kus - 1) / a.kus; // stages per row block
    const int nst = nrbc * sprb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ns; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (ARGMAX && threadIdx.x < MX)
        s_key[threadIdx.x] = 0ull;
    __syncthreads();
    pdl_launch_dependents();

    const uint32_t ring = smem_addr(smem);
    float *spart = reinterpret_cast<float *>(smem + a.off_spart);
    float *rbpart = reinterpret_cast<float *>(smem + a.off_rbpart);

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------- producer warp
        // Weights do not depend on earlier kernels, so no griddepcontrol.wait.
        const uint64_t pol = policy_evict_first();
        const int row_words = a.K >> 3, row_steps = a.K >> 5;
        for (int i = 0; i < nst; ++i) {
            const int slot = (i & (kConsumerWarps - 1)) + kConsumerWarps * ((i / kConsumerWarps) % a.dpw);
            const int use = (i / kConsumerWarps) / a.dpw;
            if (use > 0) {
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait_bounded(smem_addr(&empty_bar[slot]), (use - 1) & 1,
                                           s_abort ? kDrainLimit : kWaitLimit);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok && lane == 0) {
                    s_abort = 1;
                    atomicOr(a.err, 1);
                }
            }
            const int rbl = i / sprb, j = i - rbl * sprb;
            const int rb = rb0 + rbl;
            const int kua = ku0 + j * a.kus;
            const int nk = min(a.kus, ku0 + nkuc - kua);
            const int rows = min(16, a.N - rb * 16);
            const uint32_t qbytes = nk * 128u, sbytes = nk * 16u;
            const uint32_t bar = smem_addr(&full_bar[slot]);
            if (lane == 0)
                mbar_arrive_expect_tx(bar, rows * (qbytes + sbytes));
            __syncwarp();
            const uint32_t sb = ring + slot * a.slot_bytes;
            const int r = lane & 15;
            if (r < rows) {
                const size_t row = (size_t)rb * 16 + r;
                if (lane < 16)
                    bulk_g2s(sb + r * a.pq, a.qw + row * row_words + kua * 32, qbytes, bar, pol);
                else
                    bulk_g2s(sb + 16 * a.pq + r * a.ps, a.sc + row * row_steps + kua * 8, sbytes, bar,
                             pol);
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

        for (int i = warp; i < nst; i += kConsumerWarps) {
            const int slot = warp + kConsumerWarps * ((i / kConsumerWarps) % a.dpw);
            const int use = (i / kConsumerWarps) / a.dpw;
            if (!mbar_wait_bounded(smem_addr(&full_bar[slot]), use & 1,
                                   s_abort ? kDrainLimit : kWaitLimit)) {
                if (lane == 0) {
                    s_abort = 1;
                    atomicOr(a.err, 1);
                }
            }
            const int rbl = i / sprb, j = i - rbl * sprb;
            const int kua = ku0 + j * a.kus;
            const int nk = min(a.kus, ku0 + nkuc - kua);
            const unsigned char *sbp = smem + slot * a.slot_bytes;
            const unsigned char *qa = sbp + g * a.pq + t * 16;
            const unsigned char *qb = qa + 8 * a.pq;
            const unsigned char *pa = sbp + 16 * a.pq + g * a.ps + 4 * (t & 1);
            const unsigned char *pb = pa + 8 * a.ps;
            const uint4 *xb0 = xrow + xstep * (2 * kua);
            float accA = 0.f, accB = 0.f;
#pragma unroll 2
            for (int kt = 0; kt < 2 * nk; ++kt) {
                const uint4 wa = *reinterpret_cast<const uint4 *>(qa + kt * 64);
                const uint4 wb = *reinterpret_cast<const uint4 *>(qb + kt * 64);
                const uint32_t sa = *reinterpret_cast<const uint32_t *>(pa + kt * 8);
                const uint32_t sbv = *reinterpret_cast<const uint32_t *>(pb + kt * 8);
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
            accA += __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
            accB += __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
            const int m = t >> 1;
            if ((t & 1) == 0 && m < MX) {
                spart[(i * MX + m) * 16 + g] = accA;
                spart[(i * MX + m) * 16 + g + 8] = accB;
            }
        }
        named_sync(1, kConsumers);

        // Each row block: sum of its stages in stage order.
        for (int e = threadIdx.x; e < nrbc * MX * 16; e += kConsumers) {
            const int rr = e & 15, m = (e >> 4) % MX, rbl = e / (16 * MX);
            float s = 0.f;
            for (int j = 0; j < sprb; ++j)
                s += spart[((rbl * sprb + j) * MX + m) * 16 + rr];
            if (C == 1)
                emit<MX>(a, m, (rb0 + rbl) * 16 + rr, s, s_key, ARGMAX);
            else
                rbpart[e] = s;
        }
    }

    if (C > 1) {
        // Add the K slices of the cluster's CTAs in rank order through DSMEM;
        // rank r writes elements [r*E/C, (r+1)*E/C) of the cluster's rows.
        cluster_sync();
        if (warp < kConsumerWarps) {
            const int E = nrbc * MX * 16;
            const int e0 = (int)((long long)crank * E / C), e1 = (int)((long long)(crank + 1) * E / C);
            const uint32_t base = smem_addr(rbpart);
            for (int e = e0 + threadIdx.x; e < e1; e += kConsumers) {
                float s = 0.f;
                for (int c = 0; c < C; ++c)
                    s += ld_cluster_f32(map_rank(base + 4u * e, (uint32_t)c));
                const int rr = e & 15, m = (e >> 4) % MX, rbl = e / (16 * MX);
                emit<MX>(a, m, (rb0 + rbl) * 16 + rr, s, s_key, ARGMAX);
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

struct Geometry {
    int C = 1, nclusters = 1, kus = 1, ns = 1, dpw = 1, slot_bytes = 0, pq = 0, ps = 0;
    int off_x = 0, off_spart = 0, off_rbpart = 0, smem = 0;
    bool ok = false;
};

int ceil_div(int a, int b) { return (a + b - 1) / b; }

Geometry make_geometry(int M, int N, int K, int C, int nclusters)
{
    // Among the stage sizes and slot counts that fit the budget, keep the one
    // with the most bytes in flight (ties: larger stages).
    Geometry G;
    long long best_inflight = -1;
    const int nrb = ceil_div(N, 16), nku = K / 256;
    G.C = C;
    G.nclusters = nclusters;
    const int nkuc_max = ceil_div(nku, C);
    const int rbc_max = ceil_div(nrb, nclusters);
    const int x_bytes = M * K * 2 + 16;
    const int rbpart_bytes = (C > 1) ? rbc_max * M * 16 * 4 : 0;
    for (int dpw = 2; dpw >= 1; --dpw) {
        for (int kmax = 6; kmax >= 1; --kmax) {
            const int sprb = ceil_div(nkuc_max, kmax);
            const int kus = ceil_div(nkuc_max, sprb);
            const int pq = kus * 128 + 64, ps = kus * 16 + 16;
            const int slot_bytes = 16 * pq + 16 * ps;
            const int max_stages = rbc_max * sprb;
            const int spart_bytes = max_stages * M * 16 * 4;
            int ns = kConsumerWarps * dpw;
            if (ns > max_stages)
                ns = max_stages;
            const int off_x = ns * slot_bytes;
            const int off_spart = (off_x + x_bytes + 15) & ~15;
            const int off_rbpart = (off_spart + spart_bytes + 15) & ~15;
            const int total = off_rbpart + rbpart_bytes;
            if (total > kSmemBudget)
                continue;
            const long long inflight = (long long)ns * slot_bytes;
            if (inflight <= best_inflight)
                continue;
            best_inflight = inflight;
            G.kus = kus;
            G.pq = pq;
            G.ps = ps;
            G.slot_bytes = slot_bytes;
            G.ns = ns;
            G.dpw = dpw;
            G.off_x = off_x;
            G.off_spart = off_spart;
            G.off_rbpart = off_rbpart;
            G.smem = total;
            G.ok = true;
        }
    }
    return G;
}

template <int MX, bool ARGMAX>
cudaError_t launch_stream(const Geometry &G, const StreamArgs &a, cudaStream_t s)
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
    return cudaLaunchKernelEx(&cfg, kern, a);
}

} // namespace

bool stream_supported(int M, int N, int K, const void *qw, const void *sc)
{
    (void)N;
    return M >= 1 && M <= 2 && K % 256 == 0 && (reinterpret_cast<uintptr_t>(qw) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
}

StreamPlan plan_stream(int M, int N, int K, int num_sms)
{
    // Per-shape tiling: pick the cluster size C (K slices) and the number of
    // clusters that minimise the largest per-CTA share, one CTA per SM.
    StreamPlan best;
    const int nrb = ceil_div(N, 16), nku = K / 256;
    long long best_work = -1;
    const int cands[] = {1, 2, 3, 4, 6, 8};
    for (int C : cands) {
        if (C > nku)
            continue;
        int ncl = num_sms / C;
        if (ncl > nrb)
            ncl = nrb;
        if (ncl < 1)
            continue;
        const long long work = (long long)ceil_div(nrb, ncl) * ceil_div(nku, C);
        const Geometry G = make_geometry(M, N, K, C, ncl);
        if (!G.ok)
            continue;
        if (best_work < 0 || work < best_work) {
            best_work = work;
            best.C = C;
            best.nclusters = ncl;
        }
    }
    best.ok = best_work >= 0;
    return best;
}

cudaError_t run_stream(const StreamPlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                       const uint16_t *sc, int M, int N, int K, unsigned long long *keys,
                       int32_t *argmax, int *err, cudaStream_t s)
{
    const Geometry G = make_geometry(M, N, K, p.C, p.nclusters);
    if (!G.ok)
        return cudaErrorInvalidConfiguration;
    StreamArgs a;
    a.y = y;
    a.x = x;
    a.qw = qw;
    a.sc = sc;
    a.keys = keys;
    a.err = err;
    a.N = N;
    a.K = K;
    a.nclusters = G.nclusters;
    a.kus = G.kus;
    a.ns = G.ns;
    a.dpw = G.dpw;
    a.slot_bytes = G.slot_bytes;
    a.pq = G.pq;
    a.ps = G.ps;
    a.off_x = G.off_x;
    a.off_spart = G.off_spart;
    a.off_rbpart = G.off_rbpart;
    const bool am = argmax != nullptr;
    cudaError_t e;
    if (M == 1)
        e = am ? launch_stream<1, true>(G, a, s) : launch_stream<1, false>(G, a, s);
    else
        e = am ? launch_stream<2, true>(G, a, s) : launch_stream<2, false>(G, a, s);
    if (e != cudaSuccess || !am)
        return e;
    return run_argmax_finalize(argmax, keys, M, G.C * G.nclusters, s);
}

} // namespace w4
