/*
 * w4a16.h - C ABI of the W4A16 group-quantized GEMV/GEMM library (libw4a16.so).
 *
 * Weight format (source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch",
 * checkpoint paragraph: compressed-tensors W4A16, 4-bit weights in groups of 32
 * along K, 16-bit activations, each group's step stored in bf16; w4gemv
 * paragraph: a code c stands for (c - 8) * step, the "subtract 2^23 + 8" unpack):
 *
 *   qweight  uint32 [N][K/8]      8 codes per word along K, low nibble first:
 *                                 code (n,k) = (qweight[n][k/8] >> 4*(k%8)) & 0xF
 *   scales   bf16   [N][K/group]  raw bf16 bits (uint16_t), row-major
 *   x        bf16   [M][K]        raw bf16 bits, row-major
 *   y        fp32   [M][N]        y[m][n] = sum_k x[m][k] * (code(n,k) - 8) * scale(n, k/group)
 *
 * Conventions for every call below:
 *   - Every array pointer is a DEVICE pointer owned by the caller. The library
 *     never frees, retains or reallocates caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls only enqueue work on `stream` and return; nothing is
 *     complete until the caller synchronizes that stream.
 *   - Arguments are validated on the host before anything is launched. A call
 *     that returns an error launched nothing.
 *   - Results are bitwise deterministic run to run (no floating-point atomics).
 *   - All calls are safe to capture in a CUDA graph once the library has been
 *     initialised on the device (w4_init, or any earlier call on that device).
 *   - group is 32, 64, 128, 256 or 512 codes per step along K (32 is the
 *     checkpoint paragraph's format; the "fastgemma-gemma-4-E2B" model card's
 *     file table stores FFN and LM-head weights with group 256, the per-layer
 *     table with group 64, and mentions a group-512 build); K % group == 0.
 *   - K must be a positive multiple of 32; N and M positive; N*K/8 and M*K must
 *     fit in int32 index space as stated per call.
 *   - Pointers must be 16-byte aligned (128-bit loads); y must be 4-byte aligned.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,  /* NULL pointer, size <= 0, K % group != 0, size overflow */
    W4_ERR_UNSUPPORTED = 2,  /* group not in {32, 64, 128, 256, 512}, M beyond what the call serves */
    W4_ERR_MISALIGNED = 3,   /* a pointer is not aligned as stated above */
    W4_ERR_CUDA = 4,         /* the CUDA runtime reported an error (launch or allocation) */
    W4_ERR_NO_DEVICE = 5     /* no usable sm_103 device is current */
} w4_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char *w4_status_string(int status);

/* The CUDA error string behind the last W4_ERR_CUDA on this thread ("" if none). */
const char *w4_last_cuda_error(void);

/*
 * Set up the library on the current device: checks that it is sm_103 and
 * allocates the library-owned device scratch (4 MB of argmax keys and one
 * error word, held until process exit). Idempotent and thread-safe. Call it
 * before capturing any call of this library in a CUDA graph; otherwise the
 * first call on a device does it.
 */
int w4_init(void);

/*
 * Reads and clears the device error word of the current device after a
 * cudaDeviceSynchronize. *code is 0 when every kernel finished normally. A set
 * bit means that a kernel's bounded wait on its own shared-memory pipeline ran
 * out: bit 0 the streaming decode kernel, bit 1 the prefill GEMM, bit 2 the
 * self-test below. That kernel then returned without hanging; its outputs are
 * not valid, and the context stays usable.
 */
int w4_device_error(int32_t *code);

/*
 * Self-test of the failure path: launches one kernel on `stream` whose bounded
 * wait on an mbarrier that nothing arrives at gives up (after at most ~1 ms)
 * and sets bit 2 of the device error word, exactly as a kernel whose pipeline
 * stalled sets its bit and returns. Returns W4_OK when the launch succeeded.
 */
int w4_selftest_wait_timeout(void *stream);

/*
 * W4A16 matrix-vector product for decode, M in [1, 8].
 * Source: the w4gemv paragraph (one vector times every weight matrix; packed
 * words read directly, unpacked in registers, never a 16-bit copy) and the
 * per-shape tiling paragraph (a fixed tiling per weight shape).
 *   y [M][N] fp32 out; x [M][K] bf16; qweight [N][K/8]; scales [N][K/32].
 * The library picks the tiling from (M, N, K). Returns W4_ERR_UNSUPPORTED for
 * M > 8 (use w4a16_gemm). The kernel honours programmatic dependent launch:
 * it starts streaming weights before the previous kernel on `stream` has
 * finished and reads x only after it has.
 */
int w4a16_gemv(float *y, const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
               int M, int N, int K, int group, void *stream);

/*
 * W4A16 GEMM for any M >= 1. M <= 8 runs the decode kernel of w4a16_gemv; larger
 * M (prompt reads, the prefill paragraph: a prompt is read in chunks and every
 * weight multiplies the whole chunk) runs a tensor-core kernel that dequantizes
 * each weight tile to bf16 (round to nearest even) on its way into shared
 * memory and accumulates in fp32 in tensor memory. Same layouts as w4a16_gemv.
 * For M > 8, N must be a multiple of 16 and K a multiple of 64.
 */
int w4a16_gemm(float *y, const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
               int M, int N, int K, int group, void *stream);

/*
 * Decode GEMV with a fused greedy pick, M in [1, 8].
 * Source: Step 2 (the tied 4-bit embedding doubles as the output layer) and the
 * scope note (greedy decoding): y as w4a16_gemv, and argmax[m] = the lowest n
 * with y[m][n] equal to the largest y[m][:] (-0 and +0 compare equal; y is the
 * fp32 value written to y). argmax is a device int32 [M].
 * Uses the library-owned scratch set up by w4_init; calls that overlap in time on
 * different streams share it and must not run concurrently.
 */
int w4a16_gemv_argmax(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                      const uint16_t *scales, int M, int N, int K, int group, void *stream);

/*
 * w4a16_gemv_argmax for callers that cannot allocate device memory: a plug-in
 * loaded into a host process that owns every device allocation through its own
 * allocator, or a real-time decode loop that must not reach the driver's
 * allocator once it has started. The pages have no counterpart; this is a
 * library convenience.
 * Same arguments, layouts, results and errors as w4a16_gemv_argmax, and it runs
 * the register-streaming decode kernels. It calls no cudaMalloc/cudaFree: its
 * scratch is a fixed 256 KiB array in the library's device image (held by every
 * GPU that loads the library until exit), with room for M * CTAs <= 32768 keys;
 * a larger call (about M * N / 128 > 32768) returns W4_ERR_UNSUPPORTED.
 * The first call on a device does a one-time set-up for that device (it looks
 * up the array's device address, with that device current); make that first
 * call before any stream capture begins.
 * All calls share the array: calls that overlap in time on the GPU (for
 * example on two streams) race on it and must be serialized by the caller.
 */
int w4a16_gemv_argmax_noalloc(float *y, int32_t *argmax, const uint16_t *x,
                              const uint32_t *qweight, const uint16_t *scales, int M, int N, int K,
                              int group, void *stream);

/*
 * 4-bit row gather (the per-layer embedding lookup on the card, Step 2).
 *   out    bf16 [M][K] out: out[t][k] = bf16_rne((code(ids[t], k) - 8) * scale)
 *   ids    int32 [M] device, row indices into the table
 *   qtable uint32 [N][K/8], scales bf16 [N][K/32]
 *   status int32 device word or NULL: an id outside [0, N) gives a zero row and,
 *          if status is not NULL, stores 1 to *status (never cleared by the library).
 * The product of a 4-bit code and a bf16 step is exact in fp32, so the output is
 * bit-exact: one rounding, to nearest even.
 */
int w4_embed_gather(uint16_t *out, const int32_t *ids, const uint32_t *qtable,
                    const uint16_t *scales, int M, int N, int K, int group,
                    int32_t *status, void *stream);

/*
 * Memory read probe (the memory-read paragraph: the card's read ceiling measured
 * by a plain sum over memory). Streams `bytes` of `buf` once and stores the sum of
 * its uint32 words mod 2^64 to *sum (device uint64). bytes must be a positive
 * multiple of 16; buf 16-byte aligned. Time it with events on `stream`.
 */
int hbm_read_probe(unsigned long long *sum, const void *buf, size_t bytes, void *stream);

/*
 * Decode GEMV with Hadamard-rotated weights (source: "fastgemma-gemma-4-E2B"
 * model card, "What is in the file": every linear weight is rotated along K,
 * W' = W H^T with H orthogonal, and a runtime fast Walsh-Hadamard transform of
 * the activation makes the product identical).
 *
 *   y[m][n] = sum_k (x H)[m][k] * (code(n,k) - 8) * scale(n, k/group)  (= x W^T)
 *
 * qweight/scales hold the rotated weight W' in the usual format; H is
 * block-diagonal over blocks of `hblock` consecutive k, each the Sylvester
 * matrix H_b[i][j] = (-1)^popcount(i & j) / sqrt(b). hblock: a power of two in
 * 2..4096 dividing K. M in 1..4. argmax: NULL, or int32 [M] receiving the lowest
 * index of each row's maximum (as w4a16_gemv_argmax). x H is formed in fp32 and
 * carried as two bf16 parts (relative 2^-18), so the decode tolerance holds.
 * For M = 1 with hblock 256 or 512, K % 128 == 0 and N below the vocabulary
 * sizes (where the large-N form takes over) the decode kernel forms x H itself
 * while it stages x (one launch, no scratch). Otherwise a separate
 * transform launch writes the rotated rows to the library's split scratch
 * (like w4a16_gemm): such calls must not run concurrently on different streams.
 * Both forms give the same bits.
 */
int w4a16_gemv_hadamard(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, int M, int N, int K, int group, int hblock, void *stream);

/*
 * Decode attention of one query token over a one-head key/value cache (source:
 * "Gemma 4 E2B on a 4 GB GPU with pure PyTorch", decode-attention paragraph: one
 * key/value head serves eight query heads and each cached key and value is read
 * once for all of them, the cache split into slices combined with an online
 * softmax; cache paragraph: full layers keep one slot per position, sliding
 * layers a ring that records each slot's position; "Step 4 - The Model in
 * Rust": a slot is kept iff its position p satisfies p >= 0, p <= qpos and,
 * when window > 0, p > qpos - window).
 *
 *   out[h][d] = sum_t w[h][t] * v[t][d],  w[h][.] = softmax over kept slots t of
 *               scale * sum_d q[h][d] * k[t][d]
 *
 *   out    fp32 [H][D] (4-byte aligned); a head with no kept slot gives zeros
 *   q      bf16 [H][D] query heads sharing the key/value head (16-byte aligned)
 *   k, v   bf16 [T][D] cache slots, slot-major (16-byte aligned)
 *   kpos   int32 [T] position recorded in each slot (-1 = empty), or NULL:
 *          slot t holds position t (a full-length cache)
 *   qpos   the query's position; window 0 = no window
 *   H in 1..8, T >= 1, D in {128, 256, 384, 512}, T * D < 2^31.
 * Precision: bf16 x bf16 products accumulated in fp32 for the scores; the
 * softmax weights are rounded to bf16 for the value product (and the
 * normalising sum adds the rounded weights); fp32 accumulation; results are
 * deterministic. Uses the library's split scratch (like w4a16_gemm): calls that
 * need it must not run concurrently on different streams.
 */
int w4_attn_decode(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *kpos, int qpos, int window, int H, int T, int D, float scale,
                   void *stream);

/*
 * Decode attention with the query position in device memory (source: "Gemma 4
 * E2B on a 4 GB GPU with pure PyTorch", CUDA-graph paragraph: a cache length
 * held as a host integer is frozen into a captured graph, so the engine keeps
 * every position on the GPU). Same operation, arguments, limits and errors as
 * w4_attn_decode, except that the query position is *qpos (int32, 4-byte
 * aligned), read when the kernels run, and `window` derives the lower bound
 * from it; one captured call serves every decode step.
 */
int w4_attn_decode_devpos(float *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *kpos, const int32_t *qpos, int window, int H, int T, int D,
                          float scale, void *stream);

/*
 * Appends the new token's key and value rows to a one-head cache at the device
 * position *pos (source: the same article's cache paragraph: full layers keep
 * one slot per position, sliding layers a ring of slots that records each
 * slot's position).
 *
 *   kpos != NULL (ring of T slots): slot = *pos mod T, kpos[slot] = *pos
 *   kpos == NULL (full cache):      slot = *pos, which must lie in [0, T)
 *   k_cache[slot][:] = k_new, v_cache[slot][:] = v_new (bf16 [D] each)
 *
 * k_cache, v_cache bf16 [T][D]; k_new, v_new bf16 [D]; all 16-byte aligned;
 * pos, kpos, status int32, 4-byte aligned. D a multiple of 8, T * D < 2^31. A
 * negative position, or one outside a full cache, writes nothing and sets
 * *status = 1 (status may be NULL). *pos is read when the kernel runs and is
 * not changed.
 */
int w4_kv_append(uint16_t *k_cache, uint16_t *v_cache, int32_t *kpos, const uint16_t *k_new,
                 const uint16_t *v_new, const int32_t *pos, int T, int D, int32_t *status, void *stream);

/*
 * Greedy LM head with a forced-token skip (source: "Gemma 4 E2B on a 4 GB GPU
 * with pure PyTorch", tool-calling paragraph: when the constrained decoder
 * admits exactly one token, the step skips the int4 LM-head read).
 *
 *   *forced <  0: as w4a16_gemv_argmax with M = 1 (y = x W^T, argmax[0] = the
 *                 lowest index of the maximum)
 *   *forced >= 0: no weight is read, y is left as it was, argmax[0] = *forced
 *
 * forced: device int32 (4-byte aligned). The decode kernel reads it when it
 * starts, before it waits on the kernel preceding it on the stream (its weight
 * loads begin at launch), so *forced must hold this step's value before that
 * preceding kernel starts: write it with a copy issued ahead of the step's
 * kernels, as a host-side constrained decoder does, not from the kernel right
 * before this call. Arguments and errors otherwise as w4a16_gemv_argmax.
 */
int w4a16_gemv_argmax_forced(float *y, int32_t *argmax, const uint16_t *x, const uint32_t *qweight,
                             const uint16_t *scales, int N, int K, int group, const int32_t *forced,
                             void *stream);

/*
 * Next-step prologue of a device-resident decode loop (source: "Gemma 4 E2B on
 * a 4 GB GPU with pure PyTorch": the CUDA-graph paragraph, with every position
 * on the GPU; the emb4 paragraph, in which the embedding and the LM head share
 * one 4-bit table; Step 2, in which the row lookup happens on the card).
 *
 *   tok = *token                      (the LM head's argmax, or the forced token)
 *   tokens[*pos + 1] = tok            (when tokens != NULL and *pos + 1 in [0, cap))
 *   *pos = *pos + 1
 *   x_next[k] = bf16_rne((code(tok, k) - 8) * scale(tok, k/group))  (as w4_embed_gather)
 *
 * qtable uint32 [V][K/8], scales bf16 [V][K/group] (the 4-bit table, group 32,
 * 64, 128, 256 or 512); x_next bf16 [K] (16-byte aligned); pos, token, tokens,
 * status int32 (4-byte aligned). A token outside [0, V) gives a zero row and
 * sets bit 0 of *status; a full history sets bit 1 (status may be NULL; bits
 * are only ever set). The position is read and written when the kernel runs;
 * it must stay below 2^31 - 1 (the increment is not checked for overflow).
 */
int w4_decode_prologue(uint16_t *x_next, int32_t *tokens, int32_t *pos, const int32_t *token,
                       const uint32_t *qtable, const uint16_t *scales, int V, int K, int group, int cap,
                       int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
