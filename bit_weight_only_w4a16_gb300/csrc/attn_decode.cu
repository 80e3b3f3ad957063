// Decode attention of one query token over a one-head key/value cache.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the decode-attention
// paragraph (one key/value head serves eight query heads, so each cached key
// and value is read once for all eight; the cache is split into slices whose
// partial results are combined with an online softmax) and the cache paragraph
// (full layers: one slot per position, one head of width 512; sliding layers:
// a 512-slot ring recording each slot's position); "Step 4 - The Model in
// Rust" (a slot is kept only if its position is >= 0, not after the query and,
// with a window w, after the query's position minus w).
//
// GB300 design. The cache is read once (T * D * 4 bytes for keys and values),
// so the kernel is bound by HBM reads; the eight heads give 4 multiply-adds per
// cached byte, which the warp-level tensor core absorbs:
//   - a CTA owns a contiguous slice of 16-token tiles; warp w owns head dims
//     [128 w, 128 w + 128) and streams its own bytes of each tile (keys and
//     values) through a 3-tile shared-memory ring with per-thread cp.async, so
//     no CTA-wide synchronisation guards the ring. Masked and out-of-range
//     slots are zero-filled instead of read;
//   - scores: m16n8k16 bf16 mma with the 16 tokens as rows and the 8 query
//     heads as the 8 columns (A from the swizzled key tile via ldmatrix, B the
//     query held in registers), fp32 accumulation in two chains; the warps'
//     partial scores (their head-dim slices) are added through shared memory
//     in warp order, so every warp sees bit-identical scores;
//   - online softmax in the exp2 domain per head; each weight goes to the
//     value product as two bf16 parts (hi = bf16(p), lo = bf16(p - hi): within
//     2^-18 of p, against 2^-9 for one bf16) and the running sum adds exactly
//     those applied weights, so the normalisation matches them;
//   - values: two mmas (the weights' hi and lo parts) with the warp's 16 head
//     dims as rows and the 8 heads as columns (A = value tile transposed by
//     ldmatrix.trans, B = the weights);
//   - each CTA stores its unnormalised output with its running max and sum; a
//     second kernel merges the slices in a fixed order (deterministic);
//   - the query position may live in device memory ("with every position on
//     the GPU", the cache paragraph): it is read after the wait on the previous
//     kernel, so one captured graph serves every decode step. Without a slot
//     table (slot t holds position t) a CTA drops the tiles that hold no kept
//     position; such tiles add nothing (zero weights, unchanged running max),
//     so the result is bitwise the same as streaming them.
// Shared-memory tiles are [16 tokens][128 dims] with 16-byte chunk c of row r
// stored at chunk c ^ (r & 7), so both ldmatrix forms read conflict-free.
#include "common.cuh"
#include "internal.h"

#include <cuda_bf16.h>

namespace w4 {

namespace {

constexpr int kTok = 16;                     // tokens per tile
constexpr int kDW = 128;                     // head dims per warp
constexpr int kHalf = kTok * kDW * 2;        // key (or value) bytes of one tile for one warp
constexpr int kSlot = 2 * kHalf;             // keys then values
constexpr int kHeads = 8;                    // query heads per key/value head (mma columns)

struct AttnArgs {
    const uint16_t *q, *k, *v;
    const int32_t *kpos;
    float *ws_o;  // [nsplit][8][D] unnormalised outputs
    float *ws_ml; // [nsplit][8][2] running max (log2 domain) and sum
    long long qpos, lo; // kept positions: lo < p <= qpos (lo = -1 without a window)
    const int32_t *qpos_dev; // when set: qpos = *qpos_dev at run time, lo from `window`
    long long window;
    int H, T, D, ntiles;
    float scale_log2; // scale * log2(e)
};

__device__ __forceinline__ bool slot_kept(const AttnArgs &a, int tok, long long qpos, long long lo)
{
    if (tok >= a.T)
        return false;
    const long long p = a.kpos ? (long long)__ldg(a.kpos + tok) : (long long)tok;
    return p >= 0 && p <= qpos && p > lo;
}

// 16-byte cp.async that writes zeros instead of reading when !valid.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// Two fp32 values rounded to bf16 (nearest even), the first in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

// GR groups of NW warps per CTA: group gi streams the gi-th half of the CTA's
// tiles with its own online-softmax state; the groups' states are merged in
// shared memory so the CTA stores one slice partial.
template <int NW, int kRing, int GR>
__global__ void __launch_bounds__(GR * NW * 32)
attn_split_kernel(const AttnArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int gi = w / NW, wl = w - gi * NW; // group, warp within the group
    const int g = lane >> 2, tq = lane & 3;
    const uint32_t ring = smem_addr(smem) + w * kRing * kSlot;
    // [GR][2][NW][16 tokens][8 heads]
    float *sp = reinterpret_cast<float *>(smem + GR * NW * kRing * kSlot) + gi * 2 * NW * 128;
    const int ctile0 = (int)((long long)blockIdx.x * a.ntiles / gridDim.x);
    const int cnt = (int)((long long)(blockIdx.x + 1) * a.ntiles / gridDim.x) - ctile0;
    const int nt0 = (cnt + 1) >> 1;
    int tile0 = GR == 1 ? ctile0 : ctile0 + (gi ? nt0 : 0);
    int nt = GR == 1 ? cnt : (gi ? cnt - nt0 : nt0);
    const int d0 = wl * kDW;

    pdl_launch_dependents();
    pdl_wait(); // the query, the cache and the position may be written by the previous kernel

    long long qpos = a.qpos, lo = a.lo;
    if (a.qpos_dev != nullptr) {
        qpos = (long long)*a.qpos_dev;
        lo = a.window > 0 ? qpos - a.window : -1;
    }
    if (a.kpos == nullptr) {
        // Kept slots lie in [lo + 1, min(qpos, T - 1)]: only tiles [ft, et) hold any.
        const long long last = qpos < (long long)a.T - 1 ? qpos : (long long)a.T - 1;
        const long long ft = lo < 0 ? 0 : (lo + 1) / kTok;
        const long long et = last < 0 ? 0 : last / kTok + 1;
        const long long b = tile0 > ft ? tile0 : ft;
        const long long e = (long long)tile0 + nt < et ? (long long)tile0 + nt : et;
        tile0 = (int)(b < e ? b : tile0);
        nt = (int)(b < e ? e - b : 0);
    }

    // Query as the score mma's B operand: head g, dims d0 + 16 s + 2 tq (+1) and + 8 (+9).
    uint32_t qb[8][2];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const bool ok = g < a.H;
        const uint16_t *qp = a.q + (size_t)g * a.D + d0 + 16 * s + 2 * tq;
        qb[s][0] = ok ? ldg_nc_u32(qp) : 0u;
        qb[s][1] = ok ? ldg_nc_u32(qp + 8) : 0u;
    }

    // Copies this warp's 128 dims of tile i (relative to tile0) into ring slot
    // `slot`; one commit group per call (empty past the end).
    auto issue = [&](int i, int slot) {
        if (i < nt) {
            const int tb = (tile0 + i) * kTok;
            const uint32_t kb = ring + slot * kSlot;
#pragma unroll
            for (int c = lane; c < kTok * 16; c += 32) {
                const int r = c >> 4, j = c & 15;
                const bool ok = slot_kept(a, tb + r, qpos, lo);
                const size_t off = (size_t)(ok ? tb + r : 0) * a.D + d0 + j * 8;
                const uint32_t so = r * 256 + ((j ^ (r & 7)) << 4);
                cp_async16_zfill(kb + so, a.k + off, ok);
                cp_async16_zfill(kb + kHalf + so, a.v + off, ok);
            }
        }
        cp_async_commit_group();
    };

#pragma unroll
    for (int i = 0; i < kRing - 1; ++i)
        issue(i, i);

    float m_run = -INFINITY, l_run = 0.f; // head g, log2 domain
    float o[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s)
        o[s][0] = o[s][1] = o[s][2] = o[s][3] = 0.f;

    for (int i = 0; i < nt; ++i) {
        issue(i + kRing - 1, (i + kRing - 1) % kRing);
        cp_async_wait_group<kRing - 1>();
        __syncwarp(); // every lane's copies of tile i are in place
        const uint32_t kb = ring + (i % kRing) * kSlot, vb = kb + kHalf;

        // Partial scores S[token][head] over this warp's dims: two chains.
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mi = lane >> 3, row = (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const int ch = 2 * s + (mi >> 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + row * 256 + ((ch ^ (row & 7)) << 4), a0, a1, a2, a3);
                mma_16816((s & 1) ? c1 : c0, a0, a1, a2, a3, qb[s][0], qb[s][1]);
            }
        }
        float *spb = sp + (i & 1) * NW * 128;
        {
            float *mine = spb + wl * 128;
            mine[g * 8 + 2 * tq] = c0[0] + c1[0];
            mine[g * 8 + 2 * tq + 1] = c0[1] + c1[1];
            mine[(g + 8) * 8 + 2 * tq] = c0[2] + c1[2];
            mine[(g + 8) * 8 + 2 * tq + 1] = c0[3] + c1[3];
        }
        if (NW > 1)
            named_sync(1 + gi, NW * 32);
        else
            __syncwarp();

        // Scores of head g for tokens 2tq, 2tq+1, 2tq+8, 2tq+9 (this lane's
        // share of the value mma's B operand), added in warp order.
        const int tb = (tile0 + i) * kTok;
        float sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = 2 * tq + (j & 1) + 8 * (j >> 1);
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < NW; ++u)
                acc += spb[u * 128 + tok * 8 + g];
            sc[j] = slot_kept(a, tb + tok, qpos, lo) ? acc * a.scale_log2 : -INFINITY;
        }
        float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);
        float alpha = 1.f, p[4] = {0.f, 0.f, 0.f, 0.f};
        if (m_new != -INFINITY) {
            alpha = exp2f(m_run - m_new); // 0 while nothing was kept before
#pragma unroll
            for (int j = 0; j < 4; ++j)
                p[j] = exp2f(sc[j] - m_new); // 0 for masked slots
        }
        // Each weight as two bf16 parts, hi = bf16(p) and lo = bf16(p - hi) (p - hi
        // is exact in fp32): the value product applies hi + lo, within 2^-18 of
        // p, and hi + lo is exact in fp32 (at most 17 significant bits), so the
        // running sum adds exactly the weights applied.
        const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
        const float h0 = bf16lo_to_f32(pb0), h1 = bf16hi_to_f32(pb0);
        const float h2 = bf16lo_to_f32(pb1), h3 = bf16hi_to_f32(pb1);
        const uint32_t pl0 = pack_bf16(p[0] - h0, p[1] - h1), pl1 = pack_bf16(p[2] - h2, p[3] - h3);
        float psum = (h0 + bf16lo_to_f32(pl0)) + (h1 + bf16hi_to_f32(pl0)) + (h2 + bf16lo_to_f32(pl1)) +
                     (h3 + bf16hi_to_f32(pl1));
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 1);
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 2);
        l_run = l_run * alpha + psum;
        m_run = m_new;

        // Rescale the running outputs of heads 2tq, 2tq+1 (their alphas live on
        // lanes 8tq and 8tq+4), then add this tile's values.
        const float al0 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * tq);
        const float al1 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * tq + 4);
        {
            const int mi = lane >> 3, row = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                o[s][0] *= al0;
                o[s][1] *= al1;
                o[s][2] *= al0;
                o[s][3] *= al1;
                const int ch = 2 * s + (mi & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb + row * 256 + ((ch ^ (row & 7)) << 4), a0, a1, a2, a3);
                mma_16816(o[s], a0, a1, a2, a3, pb0, pb1);
                mma_16816(o[s], a0, a1, a2, a3, pl0, pl1);
            }
        }
    }
    cp_async_wait_group<0>(); // only empty groups remain

    if (GR == 2) {
        // Group 1 leaves its state in its own (finished) ring; group 0 merges:
        // m = max(m0, m1), each side scaled by 2^(m_i - m).
        float *park = reinterpret_cast<float *>(smem + (size_t)(NW + wl) * kRing * kSlot) + lane * 34;
        if (gi == 1) {
#pragma unroll
            for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    park[s2 * 4 + c] = o[s2][c];
            park[32] = m_run;
            park[33] = l_run;
        }
        __syncthreads();
        if (gi == 1)
            return;
        const float m1 = park[32], l1 = park[33];
        const float mm = fmaxf(m_run, m1);
        const float f0 = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mm);
        const float f1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - mm);
        l_run = l_run * f0 + l1 * f1;
        m_run = mm;
        // o holds heads 2tq, 2tq+1, whose factors live on lanes 8tq and 8tq+4.
        const float a0 = __shfl_sync(0xFFFFFFFFu, f0, 8 * tq), a1 = __shfl_sync(0xFFFFFFFFu, f0, 8 * tq + 4);
        const float b0 = __shfl_sync(0xFFFFFFFFu, f1, 8 * tq), b1 = __shfl_sync(0xFFFFFFFFu, f1, 8 * tq + 4);
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
            o[s2][0] = o[s2][0] * a0 + park[s2 * 4 + 0] * b0;
            o[s2][1] = o[s2][1] * a1 + park[s2 * 4 + 1] * b1;
            o[s2][2] = o[s2][2] * a0 + park[s2 * 4 + 2] * b0;
            o[s2][3] = o[s2][3] * a1 + park[s2 * 4 + 3] * b1;
        }
    }

    // Unnormalised slice outputs, running max and sum (heads >= H are unused).
    float *wo = a.ws_o + (size_t)blockIdx.x * kHeads * a.D;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const int d = d0 + 16 * s + g;
        wo[(size_t)(2 * tq) * a.D + d] = o[s][0];
        wo[(size_t)(2 * tq + 1) * a.D + d] = o[s][1];
        wo[(size_t)(2 * tq) * a.D + d + 8] = o[s][2];
        wo[(size_t)(2 * tq + 1) * a.D + d + 8] = o[s][3];
    }
    if (wl == 0 && tq == 0) {
        a.ws_ml[((size_t)blockIdx.x * kHeads + g) * 2] = m_run;
        a.ws_ml[((size_t)blockIdx.x * kHeads + g) * 2 + 1] = l_run;
    }
}

// out[h][d] = sum_s O_s[h][d] 2^(m_s - m) / sum_s l_s 2^(m_s - m) with m the
// largest m_s. Block (32 dims, head), one pass: warp w merges the slices
// s = w, w + 8, ... in that order into a running (max, sum, output) for its
// lane's dim, four slices' loads in flight at a time; warp 0 then merges the 8
// warp states in warp order (deterministic). A slice that kept no slot
// (m_s = -inf) adds nothing.
constexpr int kCombWarps = 8;
constexpr int kCombBatch = 4;

__device__ __forceinline__ void merge_state(float &M, float &L, float &O, float m, float l, float o)
{
    if (m == -INFINITY)
        return;
    const float Mn = fmaxf(M, m);
    const float a = exp2f(M - Mn); // 0 while nothing was merged (M = -inf)
    const float b = exp2f(m - Mn);
    L = fmaf(L, a, l * b);
    O = fmaf(O, a, o * b);
    M = Mn;
}

__global__ void __launch_bounds__(kCombWarps * 32)
attn_combine_kernel(float *__restrict__ out, const float *__restrict__ ws_o, const float *__restrict__ ws_ml,
                    int nsplit, int D)
{
    __shared__ float sm[kCombWarps], sl[kCombWarps], so[kCombWarps][32];
    pdl_wait();
    const int h = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int d = blockIdx.x * 32 + lane;
    const bool dok = d < D;

    float M = -INFINITY, L = 0.f, O = 0.f;
    for (int s0 = w; s0 < nsplit; s0 += kCombBatch * kCombWarps) {
        float mv[kCombBatch], lv[kCombBatch], ov[kCombBatch];
#pragma unroll
        for (int j = 0; j < kCombBatch; ++j) {
            const int sidx = s0 + j * kCombWarps;
            const bool ok = sidx < nsplit;
            const size_t r = (size_t)(ok ? sidx : 0) * kHeads + h;
            mv[j] = ok ? ws_ml[r * 2] : -INFINITY;
            lv[j] = ok ? ws_ml[r * 2 + 1] : 0.f;
            ov[j] = (ok && dok) ? ws_o[r * D + d] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kCombBatch; ++j)
            merge_state(M, L, O, mv[j], lv[j], ov[j]);
    }
    if (lane == 0) {
        sm[w] = M;
        sl[w] = L;
    }
    so[w][lane] = O;
    __syncthreads();
    if (w == 0 && dok) {
        float Mt = -INFINITY, Lt = 0.f, Ot = 0.f;
#pragma unroll
        for (int u = 0; u < kCombWarps; ++u)
            merge_state(Mt, Lt, Ot, sm[u], sl[u], so[u][lane]);
        out[(size_t)h * D + d] = (Mt != -INFINITY && Lt > 0.f) ? Ot / Lt : 0.f;
    }
}

template <int NW>
cudaError_t launch_attn(const AttnArgs &a0, float *out, float *ws, size_t ws_floats, int num_sms,
                        cudaStream_t s)
{
    // Ring depth 3: two CTAs (8 warps) per SM at D = 512. Measured at 131072
    // slots x 512: depth 2 / 3 / 4 / 6 (3 / 2 / 1 / 1 CTAs per SM) took
    // 53.4 / 50.5 / 67.7 / 69.9 us; warps per SM matter more than depth.
    constexpr int R = 3;
    constexpr int GR = NW == 4 ? 2 : 1; // one CTA of 8 warps per SM at D = 512
    auto kern = attn_split_kernel<NW, R, GR>;
    const size_t smem = (size_t)GR * NW * R * kSlot + (size_t)GR * 2 * NW * 128 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, GR * NW * 32, smem);
    if (e != cudaSuccess)
        return e;
    if (occ < 1)
        return cudaErrorInvalidConfiguration;
    // One resident wave of slices; every slice at least one tile; partials fit ws.
    int nsplit = num_sms * occ;
    if (nsplit > a0.ntiles)
        nsplit = a0.ntiles;
    const size_t per = (size_t)kHeads * a0.D + 2 * kHeads;
    if ((size_t)nsplit * per > ws_floats)
        nsplit = (int)(ws_floats / per);
    if (nsplit < 1)
        return cudaErrorInvalidValue;
    AttnArgs a = a0;
    a.ws_o = ws;
    a.ws_ml = ws + (size_t)nsplit * kHeads * a0.D;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsplit);
    cfg.blockDim = dim3(GR * NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess)
        return e;

    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(a0.D / 32, a0.H);
    cfg2.blockDim = dim3(kCombWarps * 32);
    cfg2.dynamicSmemBytes = 0;
    cfg2.stream = s;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, attn_combine_kernel, out, (const float *)a.ws_o, (const float *)a.ws_ml,
                              nsplit, a0.D);
}

} // namespace

cudaError_t run_attn_decode(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int32_t *kpos, long long qpos, const int32_t *qpos_dev, long long window,
                            int H, int T, int D, float scale, float *ws, size_t ws_floats, int num_sms,
                            cudaStream_t s)
{
    AttnArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.kpos = kpos;
    a.qpos = qpos;
    a.lo = window > 0 ? qpos - window : -1;
    a.qpos_dev = qpos_dev;
    a.window = window;
    a.H = H;
    a.T = T;
    a.D = D;
    a.ntiles = (T + kTok - 1) / kTok;
    a.scale_log2 = scale * 1.4426950408889634f;
    switch (D / kDW) {
    case 1: return launch_attn<1>(a, out, ws, ws_floats, num_sms, s);
    case 2: return launch_attn<2>(a, out, ws, ws_floats, num_sms, s);
    case 3: return launch_attn<3>(a, out, ws, ws_floats, num_sms, s);
    case 4: return launch_attn<4>(a, out, ws, ws_floats, num_sms, s);
    default: return cudaErrorNotSupported;
    }
}

} // namespace w4
