// Device-resident decode-step plumbing: the key/value append at the current
// position and the next-step prologue.
//
// Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the CUDA-graph
// paragraph (a decode step is captured once and replayed for every token; a
// cache length kept as a host integer is frozen into the graph, so the engine
// keeps every position on the GPU), the emb4 paragraph (the embedding and the LM
// head share one 4-bit table) and the tool-calling paragraph (a step whose
// constrained decoder admits one token skips the LM-head read; the forced-token
// form of the greedy LM head lives in gemv_decode.cu).
//
// One step on the device: kv_append (slot of *pos) -> attention reading *pos ->
// LM head (argmax, or the forced token) -> prologue (token history, *pos + 1,
// embedding row of the token as the next step's x). Nothing in it is a host
// value, so the captured graph of one step replays for every token. Both
// kernels move a few KB and are latency-bound: one CTA, 16-byte accesses.
#include "common.cuh"
#include "internal.h"

namespace w4 {

namespace {

__global__ void __launch_bounds__(128)
kv_append_kernel(uint16_t *__restrict__ kc, uint16_t *__restrict__ vc, int32_t *__restrict__ kpos,
                 const uint16_t *__restrict__ kn, const uint16_t *__restrict__ vn, const int32_t *pos, int T,
                 int D, int32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait(); // the new rows and the position may come from the previous kernel
    const long long p = *pos;
    long long slot = -1;
    if (p >= 0)
        slot = kpos != nullptr ? p % T : (p < T ? p : -1);
    if (slot < 0) {
        if (threadIdx.x == 0 && status != nullptr)
            *status = 1;
        return;
    }
    const int chunks = D >> 3; // 16-byte chunks of one row
    for (int c = threadIdx.x; c < 2 * chunks; c += blockDim.x) {
        const bool isv = c >= chunks;
        const int j = isv ? c - chunks : c;
        const uint4 val = reinterpret_cast<const uint4 *>(isv ? vn : kn)[j];
        reinterpret_cast<uint4 *>((isv ? vc : kc) + (size_t)slot * D)[j] = val;
    }
    if (kpos != nullptr && threadIdx.x == 0)
        kpos[slot] = (int32_t)p;
}

__global__ void __launch_bounds__(256)
decode_prologue_kernel(uint16_t *__restrict__ x_next, int32_t *__restrict__ tokens, int32_t *pos,
                       const int32_t *tok_in, const uint32_t *__restrict__ qt, const uint16_t *__restrict__ sc,
                       int V, int K, int lg, int cap, int32_t *__restrict__ status)
{
    pdl_launch_dependents();
    pdl_wait(); // the token is the previous kernel's output
    const int tok = *tok_in;
    const bool ok = tok >= 0 && tok < V;
    const int words = K >> 3;
    const int nsteps = K >> (5 + lg); // one step per 32 << lg codes
    for (int wd = threadIdx.x; wd < words; wd += blockDim.x) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (ok) {
            const uint32_t w = qt[(size_t)tok * words + wd];
            const float s = bf16lo_to_f32(sc[(size_t)tok * nsteps + ((wd >> 2) >> lg)]);
            o.x = bf16x2_of_codes(w, 0, s);
            o.y = bf16x2_of_codes(w, 8, s);
            o.z = bf16x2_of_codes(w, 16, s);
            o.w = bf16x2_of_codes(w, 24, s);
        }
        reinterpret_cast<uint4 *>(x_next)[wd] = o;
    }
    if (threadIdx.x == 0) {
        const long long nx = (long long)*pos + 1;
        int st = ok ? 0 : 1;
        if (tokens != nullptr) {
            if (nx >= 0 && nx < cap)
                tokens[nx] = tok;
            else
                st |= 2;
        }
        *pos = (int32_t)nx;
        if (st != 0 && status != nullptr)
            *status |= st;
    }
}

cudaLaunchConfig_t one_cta(unsigned threads, cudaStream_t s, cudaLaunchAttribute *attr)
{
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

} // namespace

cudaError_t run_kv_append(uint16_t *kc, uint16_t *vc, int32_t *kpos, const uint16_t *kn, const uint16_t *vn,
                          const int32_t *pos, int T, int D, int32_t *status, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = one_cta(128, s, attr);
    return cudaLaunchKernelEx(&cfg, kv_append_kernel, kc, vc, kpos, kn, vn, pos, T, D, status);
}

cudaError_t run_decode_prologue(uint16_t *x_next, int32_t *tokens, int32_t *pos, const int32_t *argmax,
                                const uint32_t *qt, const uint16_t *sc, int V, int K, int lg, int cap,
                                int32_t *status, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = one_cta(256, s, attr);
    return cudaLaunchKernelEx(&cfg, decode_prologue_kernel, x_next, tokens, pos, argmax, qt, sc, V, K, lg, cap,
                              status);
}

} // namespace w4
