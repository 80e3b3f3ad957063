// 4-bit row gather: the per-layer embedding lookup done on the card.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch", Step 2 - Keep the
// Vocabulary Tables in 4-Bit: the embedding and the per-layer table are stored as
// 4-bit codes with a 16-bit step per group, and the per-layer row lookup happens
// on the card.
//
// out[t][k] = bf16_rne((code(ids[t], k) - 8) * step). A 4-bit integer times a
// bf16 step has at most 12 significant bits, so the fp32 product is exact and
// the single rounding is the conversion to bf16 (round to nearest even).
//
// One thread turns one packed word (8 codes) into 8 bf16 (16 B store); a warp
// covers 32 consecutive words of one row, so loads and stores are coalesced.
// With a 16-byte-aligned table a thread takes a whole 32-code group instead.
// The work is latency-bound at decode sizes (8 ids x 5 KB), so the grid is just
// large enough to cover the rows.
#include "common.cuh"
#include "internal.h"

#include <cuda_bf16.h>

namespace w4 {

__global__ void __launch_bounds__(256)
embed_gather_kernel(uint16_t *__restrict__ out, const int32_t *__restrict__ ids,
                    const uint32_t *__restrict__ qt, const uint16_t *__restrict__ sc, int M,
                    int N, int K, int lg, int32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int words = K >> 3;
    const int nsteps = K >> (5 + lg); // one step per 32 << lg codes
    const long long total = (long long)M * words;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int tkn = (int)(i / words);
        const int wd = (int)(i - (long long)tkn * words);
        const int id = ids[tkn];
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (id >= 0 && id < N) {
            const uint32_t w = qt[(size_t)id * words + wd];
            const float s = bf16lo_to_f32(sc[(size_t)id * nsteps + ((wd >> 2) >> lg)]);
            // codes 0..7 of the word are k = 8*wd + 0..7, low nibble first
            o.x = bf16x2_of_codes(w, 0, s);
            o.y = bf16x2_of_codes(w, 8, s);
            o.z = bf16x2_of_codes(w, 16, s);
            o.w = bf16x2_of_codes(w, 24, s);
        } else if (status != nullptr && wd == 0) {
            *status = 1;
        }
        *reinterpret_cast<uint4 *>(out + (size_t)tkn * K + 8 * wd) = o;
    }
}

// The same gather with one thread per 32-code group (four packed words, one
// 16-byte load, four 16-byte stores) when the table is 16-byte aligned: a
// quarter of the threads and of the load instructions for the same bytes (K %
// 32 == 0, so a row holds whole groups).
__global__ void __launch_bounds__(256)
embed_gather_v4_kernel(uint16_t *__restrict__ out, const int32_t *__restrict__ ids,
                       const uint32_t *__restrict__ qt, const uint16_t *__restrict__ sc, int M,
                       int N, int K, int lg, int32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int words = K >> 3, gpr = K >> 5; // words and 32-code groups per row
    const int nsteps = K >> (5 + lg);
    const long long total = (long long)M * gpr;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int tkn = (int)(i / gpr);
        const int gq = (int)(i - (long long)tkn * gpr);
        const int id = ids[tkn];
        uint4 o[4];
        if (id >= 0 && id < N) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qt + (size_t)id * words + 4 * gq);
            const float st = bf16lo_to_f32(sc[(size_t)id * nsteps + (gq >> lg)]);
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o[j].x = bf16x2_of_codes(wv[j], 0, st);
                o[j].y = bf16x2_of_codes(wv[j], 8, st);
                o[j].z = bf16x2_of_codes(wv[j], 16, st);
                o[j].w = bf16x2_of_codes(wv[j], 24, st);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[j] = make_uint4(0u, 0u, 0u, 0u);
            if (status != nullptr && gq == 0)
                *status = 1;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)tkn * K + 32 * gq);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dst[j] = o[j];
    }
}

cudaError_t run_embed_gather(uint16_t *out, const int32_t *ids, const uint32_t *qt,
                             const uint16_t *sc, int M, int N, int K, int lg, int32_t *status,
                             cudaStream_t s)
{
    const bool v4 = (reinterpret_cast<uintptr_t>(qt) & 15) == 0;
    const long long total = (long long)M * (K >> (v4 ? 5 : 3));
    long long blocks = (total + 255) / 256;
    if (blocks > 65535)
        blocks = 65535;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, v4 ? embed_gather_v4_kernel : embed_gather_kernel, out, ids, qt, sc, M, N,
                              K, lg, status);
}

} // namespace w4
