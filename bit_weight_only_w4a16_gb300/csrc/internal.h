// Internal host-side interfaces between the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace w4 {

// log2(group / 32) for the served group sizes 32, 64, 128, 256, 512; -1 otherwise.
inline int group_shift(int group)
{
    for (int lg = 0; lg <= 4; ++lg)
        if (group == (32 << lg))
            return lg;
    return -1;
}

// Per-shape launch plan of the decode kernels (M <= 8).
struct DecodePlan {
    int kernel = 2; // 2: M <= 2 kernel (full-group 128-bit loads), 3: its persistent form for
                    // very large N, 8: M <= 8 kernel, 9: its persistent form for very large N
    int ksplit = 1; // warps of a CTA that split K for one 16-row block
    int warps = 8;  // warps per CTA
    int unroll = 4; // k-tiles (m2) or groups (m8) in flight per warp
    int grid = 1;
    int cluster = 1; // 4: the M <= 8 kernel's K quarters over clusters of 4 CTAs (ksplit is per CTA)
};

DecodePlan plan_decode(int M, int N, int K, int num_sms);
// Clusters of 4 CTAs of the M <= 8 kernel's cluster form that fit on the
// current device at once (queried once per device, then cached; 0 if the query
// fails). The device set-up calls it so that no plan queries it under capture.
int m8_cluster_capacity();
// Dynamic shared memory the decode kernel of plan p takes for (M, K).
size_t decode_smem_bytes(const DecodePlan &p, int M, int K);

// Launches the decode kernel (and, when argmax != nullptr, the argmax pass that
// reduces keys[M][plan.grid]).
// lg: log2(group / 32); scales hold one step per 32 << lg codes ([N][K >> (5 + lg)]).
// pairs: the M x-rows are M/2 (hi, lo) pairs and y has M/2 rows, each the sum of
// its pair's products (M even; M == 2 or M <= 8 by the plan's kernel).
// forced (argmax only, M <= 2 kernels): when *forced >= 0 as the kernels start,
// no weight is read, y is left as it was and argmax[m] = *forced.
// hblock (pairs, M = 2, the M <= 2 kernels, K % 128 == 0, hblock 256 or 512):
// x is ONE row and the kernel forms the (hi, lo) rows of x H itself (blocks of
// hblock) while staging x.
cudaError_t run_decode(const DecodePlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                       const uint16_t *sc, int M, int N, int K, int lg, unsigned long long *keys,
                       int32_t *argmax, cudaStream_t s, bool pairs = false,
                       const int32_t *forced = nullptr, int hblock = 0);

// M = 1 decode GEMV (K % 128 == 0, N % 16 == 0, below vocabulary sizes): a CTA
// of `warps` warps owns R 16-row blocks; K (T tiles of 128) is split into S
// sub-slices, one per warp of a row block.
struct M1Plan {
    bool ok = false;
    int R = 1, S = 1, T = 1, warps = 8, grid = 1;
};

M1Plan plan_decode_m1(int M, int N, int K, int num_sms);
cudaError_t run_decode_m1(const M1Plan &p, float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc,
                          int N, int K, int lg, cudaStream_t s);

// The driver's cuTensorMapEncodeTiled (looked up once), or null.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder();

// Vocabulary-sized M = 1 decode GEMV with the weights landed in shared memory by
// tensor copies (K % 768 == 0, K >= 1536, N % 16 == 0, at least two 16-row blocks per warp
// of a full wave, 16-byte aligned codes, and 16-byte aligned steps at group 32). With argmax != nullptr the per-CTA
// keys go to keys[0 .. num_sms) and argmax[0] receives the pick. A slot wait
// that runs out sets bit 0 of *err.
bool vocab_supported(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc);
// forced (with argmax): when *forced >= 0 as the kernel starts, no weight is
// read, y is left as it was and argmax[0] = *forced.
cudaError_t run_decode_vocab(float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int N, int K,
                             int lg, unsigned long long *keys, int32_t *argmax, int *err, int num_sms,
                             cudaStream_t s, const int32_t *forced = nullptr);

// The decode sweep's long M = 1 projections with the same shared-memory slots:
// rows per CTA when the form serves (N, K) (group 32, K % 768 == 0, N % 16 == 0,
// 16-byte aligned codes and steps, a CTA's slices within its slots), else 0.
// hblock (256 or 512; 0 for plain weights): Hadamard-rotated weights, the
// kernel forms the (hi, lo) rows of x H (blocks of hblock) while staging x.
int slab_rows_per_cta(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc, int hblock = 0);
cudaError_t run_decode_slab(int R, float *y, const uint16_t *x, const uint32_t *qw, const uint16_t *sc, int N,
                            int K, int *err, cudaStream_t s, int hblock = 0);

// Vocabulary-sized decode GEMV for 2..8 x-rows with the same shared-memory
// slots (group 32, K % 768 == 0, N % 16 == 0, at least two 16-row blocks per
// warp of a full wave, 16-byte aligned codes and steps, x staged whole in
// shared memory). With argmax != nullptr the per-(x-row, CTA) keys go to
// keys[M][grid] and argmax[m] receives the pick of x-row m.
struct Slots8Plan {
    bool ok = false;
    int W = 0, grid = 0;
    size_t smem = 0;
};
Slots8Plan plan_slots8(int M, int N, int K, int num_sms, int lg, const void *qw, const void *sc);
cudaError_t run_decode_slots8(const Slots8Plan &p, float *y, const uint16_t *x, const uint32_t *qw,
                              const uint16_t *sc, int M, int N, int K, unsigned long long *keys, int32_t *argmax,
                              int *err, cudaStream_t s);

// argmax[m] = index of the largest key in keys[m][0 .. nblocks), or *forced
// when forced != nullptr and *forced >= 0.
cudaError_t run_argmax_finalize(int32_t *argmax, const unsigned long long *keys, int M, int nblocks,
                                cudaStream_t s, const int32_t *forced = nullptr);

cudaError_t run_embed_gather(uint16_t *out, const int32_t *ids, const uint32_t *qt,
                             const uint16_t *sc, int M, int N, int K, int lg, int32_t *status,
                             cudaStream_t s);

cudaError_t run_read_probe(unsigned long long *sum, const void *buf, size_t bytes, int num_sms,
                           cudaStream_t s);

// Prefill (M > 8) tensor-core GEMM: grid persistent CTAs; the first `full`
// 128x256 tiles whole, the rest split S ways along K and added by a second
// kernel. ws holds the split partials (128*256 fp32 per split tile and split;
// capacity ws_floats).
struct PrefillPlan {
    int bn = 256;
    int S = 1;
    int full = 0;
    int grid = 1;
    bool ok = false;
};

PrefillPlan plan_prefill(int M, int N, int K, int num_sms, size_t ws_floats);
cudaError_t run_prefill(const PrefillPlan &p, float *y, const uint16_t *x, const uint32_t *qw,
                        const uint16_t *sc, int M, int N, int K, int lg, float *ws, int *err, cudaStream_t s);

// x2[2m] = bf16(v), x2[2m+1] = bf16(v - bf16(v)) for v = (x H)[m], H the block
// Sylvester-Hadamard matrix with blocks of b (a power of two dividing K), fp32.
cudaError_t run_hadamard_split(uint16_t *x2, const uint16_t *x, int M, int K, int b, cudaStream_t s);

// Launches a kernel whose bounded mbarrier wait cannot complete: it gives up
// within ~1 ms and sets bit 2 of *err.
cudaError_t run_bounded_wait_selftest(int *err, cudaStream_t s);

// Decode attention of one query token (H <= 8 query heads sharing one key/value
// head, D in {128, 256, 384, 512}) over T cache slots; split partials in ws.
// With qpos_dev != nullptr the query position is *qpos_dev, read at run time.
cudaError_t run_attn_decode(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int32_t *kpos, long long qpos, const int32_t *qpos_dev, long long window,
                            int H, int T, int D, float scale, float *ws, size_t ws_floats, int num_sms,
                            cudaStream_t s);

// Writes the new token's key and value rows into slot (*pos mod T) of a ring
// (kpos != nullptr, which records *pos there) or slot *pos of a full cache;
// a position outside the cache sets *status = 1 and writes nothing.
cudaError_t run_kv_append(uint16_t *kc, uint16_t *vc, int32_t *kpos, const uint16_t *kn, const uint16_t *vn,
                          const int32_t *pos, int T, int D, int32_t *status, cudaStream_t s);

// Next-step prologue: tok = argmax[0]; tokens[*pos + 1] = tok (when inside
// [0, cap)); *pos += 1; x_next = the bf16 row tok of the 4-bit table. A token
// outside [0, V) gives a zero row and sets status bit 0; a full history sets
// bit 1.
cudaError_t run_decode_prologue(uint16_t *x_next, int32_t *tokens, int32_t *pos, const int32_t *argmax,
                                const uint32_t *qt, const uint16_t *sc, int V, int K, int lg, int cap,
                                int32_t *status, cudaStream_t s);

} // namespace w4
