// Shared device helpers of the W4A16 CUDA library (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace w4 {

// ---------------------------------------------------------------- loads ----

// Streaming 128-bit load of weights: read-only path, not kept in L1, and L2
// asked to fetch the surrounding 256 B so the next k-tiles of the row hit L2.
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Read-only load that may stay in L1 (scales: neighbouring lanes share sectors).
__device__ __forceinline__ uint32_t ldg_nc_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ldg_nc_u64(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return (uint32_t)v;
}

// Ask L2 to fetch [p, p + bytes) from HBM without bringing it into the SM.
// p and bytes must be multiples of 16. L2 is the device's point of coherence,
// so warming it ahead of griddepcontrol.wait can never make a later load read
// stale data: a write by the previous kernel still lands in (and updates) L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------- programmatic launch ----

// Let the next kernel on the stream start launching (its own wait still
// blocks until this grid has completed and its writes are visible).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block until every prerequisite grid has completed and its memory is visible.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------- unpack ----

// Two 4-bit codes, at bits 0..3 and 16..19 of w, as an exact bf16x2 of (code - 8).
// 0x4300 | c is the bf16 of 128 + c (c fits the 7-bit mantissa); subtracting
// 136 leaves c - 8 in [-8, 7], which bf16 holds exactly. This is the bf16 form
// of the "OR into the bits of 2^23 and subtract 2^23 + 8" unpack.
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w)
{
    uint32_t t, r;
    // (w & 0x000F000F) | 0x43004300 in one three-input logic op
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x43084308u));
    return r;
}

// The four bf16x2 pairs of one packed word: nibbles (0,4), (1,5), (2,6), (3,7).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &p04, uint32_t &p15,
                                            uint32_t &p26, uint32_t &p37)
{
    p04 = nib_pair_bf16(w);
    p15 = nib_pair_bf16(w >> 4);
    p26 = nib_pair_bf16(w >> 8);
    p37 = nib_pair_bf16(w >> 12);
}

// x permuted for the B operand: one 8-code word k0..k7 pairs as
// (x0,x4) (x1,x5) (x2,x6) (x3,x7), matching unpack_word's pairs.
__device__ __forceinline__ uint4 permute_x8(uint4 in)
{
    uint4 o;
    o.x = __byte_perm(in.x, in.z, 0x5410);
    o.y = __byte_perm(in.x, in.z, 0x7632);
    o.z = __byte_perm(in.y, in.w, 0x5410);
    o.w = __byte_perm(in.y, in.w, 0x7632);
    return o;
}


// ------------------------------------------------- shared memory, TMA ----

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One potentially blocking test of an mbarrier phase: the thread sleeps until
// the phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase: false after `limit` tests of up to
// ~20 us each (never hangs).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int limit)
{
    for (int i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity, 20000u))
            return true;
    return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                 "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Named barrier over `count` threads (a subset of the CTA).
__device__ __forceinline__ void named_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------ cluster ----

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t a)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// ---------------------------------------------------------- tensor core ----

// D = A(16x16 bf16) * B(16x8 bf16) + C, fp32 accumulate (warp-level mma).
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// unpack_word of wa (row g) and wb (row g+8) followed by the two mmas of their
// 16-code halves, c += A(pairs 04, 15) * (x0, x1) and d += A(pairs 26, 37) *
// (x2, x3), written as one block so the unpacked pairs are produced directly in
// the mma's operand registers and the three constants are set once per block
// (measured on GB300: 557.7 -> 554.4 us per decode sweep, identical results).
__device__ __forceinline__ void unpack_mma2(float (&c)[4], float (&d)[4], uint32_t wa, uint32_t wb,
                                            uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3)
{
    asm("{\n"
        ".reg .b32 p0, p1, p2, p3, q0, q1, q2, q3, t, m, o, k;\n"
        "mov.b32 m, 0x000F000F;\n"
        "mov.b32 o, 0x43004300;\n"
        "mov.b32 k, 0x43084308;\n"
        "lop3.b32 p0, %8, m, o, 0xEA;\n"
        "shr.u32 t, %8, 4;\n lop3.b32 p1, t, m, o, 0xEA;\n"
        "shr.u32 t, %8, 8;\n lop3.b32 p2, t, m, o, 0xEA;\n"
        "shr.u32 t, %8, 12;\n lop3.b32 p3, t, m, o, 0xEA;\n"
        "lop3.b32 q0, %9, m, o, 0xEA;\n"
        "shr.u32 t, %9, 4;\n lop3.b32 q1, t, m, o, 0xEA;\n"
        "shr.u32 t, %9, 8;\n lop3.b32 q2, t, m, o, 0xEA;\n"
        "shr.u32 t, %9, 12;\n lop3.b32 q3, t, m, o, 0xEA;\n"
        "sub.rn.bf16x2 p0, p0, k;\n sub.rn.bf16x2 p1, p1, k;\n sub.rn.bf16x2 p2, p2, k;\n sub.rn.bf16x2 p3, p3, k;\n"
        "sub.rn.bf16x2 q0, q0, k;\n sub.rn.bf16x2 q1, q1, k;\n sub.rn.bf16x2 q2, q2, k;\n sub.rn.bf16x2 q3, q3, k;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {p0,q0,p1,q1}, {%10,%11}, {%0,%1,%2,%3};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%4,%5,%6,%7}, {p2,q2,p3,q3}, {%12,%13}, {%4,%5,%6,%7};\n"
        "}\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]), "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(x2), "r"(x3));
}

// The fp16 form of unpack_mma2, for x rows held in fp16 (exactly: see
// bf16x2_to_f16x2_exact). In fp16 a nibble fits the 10-bit mantissa at bits
// 0..3 and at bits 4..7 of each half, so one shift per word serves four pairs:
// (w & 0x000F000F) | 0x6400 halves are 1024 + c (minus 1032 leaves c - 8) and
// (w & 0x00F000F0) | 0x6400 halves are 1024 + 16 c (times 1/16 minus 72 leaves
// c - 8); both exact in fp16. Per word: 1 shift + 4 lop3 on the ALU pipe
// (against 3 + 4 in the bf16 form) and 2 sub + 2 fma on the FMA pipe.
__device__ __forceinline__ void unpack_mma2_f16(float (&c)[4], float (&d)[4], uint32_t wa, uint32_t wb,
                                                uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3)
{
    asm("{\n"
        ".reg .b32 p0, p1, p2, p3, q0, q1, q2, q3, t, u, ml, mh, o, k, s, b;\n"
        "mov.b32 ml, 0x000F000F;\n"
        "mov.b32 mh, 0x00F000F0;\n"
        "mov.b32 o, 0x64006400;\n"
        "mov.b32 k, 0x64086408;\n"
        "mov.b32 s, 0x2C002C00;\n"
        "mov.b32 b, 0xD480D480;\n"
        "lop3.b32 p0, %8, ml, o, 0xEA;\n"
        "lop3.b32 p1, %8, mh, o, 0xEA;\n"
        "shr.u32 t, %8, 8;\n"
        "lop3.b32 p2, t, ml, o, 0xEA;\n"
        "lop3.b32 p3, t, mh, o, 0xEA;\n"
        "lop3.b32 q0, %9, ml, o, 0xEA;\n"
        "lop3.b32 q1, %9, mh, o, 0xEA;\n"
        "shr.u32 u, %9, 8;\n"
        "lop3.b32 q2, u, ml, o, 0xEA;\n"
        "lop3.b32 q3, u, mh, o, 0xEA;\n"
        "sub.rn.f16x2 p0, p0, k;\n fma.rn.f16x2 p1, p1, s, b;\n sub.rn.f16x2 p2, p2, k;\n fma.rn.f16x2 p3, p3, s, b;\n"
        "sub.rn.f16x2 q0, q0, k;\n fma.rn.f16x2 q1, q1, s, b;\n sub.rn.f16x2 q2, q2, k;\n fma.rn.f16x2 q3, q3, s, b;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {p0,q0,p1,q1}, {%10,%11}, {%0,%1,%2,%3};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%4,%5,%6,%7}, {p2,q2,p3,q3}, {%12,%13}, {%4,%5,%6,%7};\n"
        "}\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]), "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(x2), "r"(x3));
}

// unpack_mma2 with both mmas chained into one accumulator: c += A(pairs 04,
// 15) * (x0, x1) + A(pairs 26, 37) * (x2, x3). For the M <= 8 slot form, where
// lane t holds word t of one 32-code group, so c is that group's partial.
__device__ __forceinline__ void unpack_mma2_1(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t x0, uint32_t x1,
                                              uint32_t x2, uint32_t x3)
{
    asm("{\n"
        ".reg .b32 p0, p1, p2, p3, q0, q1, q2, q3, t, m, o, k;\n"
        "mov.b32 m, 0x000F000F;\n"
        "mov.b32 o, 0x43004300;\n"
        "mov.b32 k, 0x43084308;\n"
        "lop3.b32 p0, %4, m, o, 0xEA;\n"
        "shr.u32 t, %4, 4;\n lop3.b32 p1, t, m, o, 0xEA;\n"
        "shr.u32 t, %4, 8;\n lop3.b32 p2, t, m, o, 0xEA;\n"
        "shr.u32 t, %4, 12;\n lop3.b32 p3, t, m, o, 0xEA;\n"
        "lop3.b32 q0, %5, m, o, 0xEA;\n"
        "shr.u32 t, %5, 4;\n lop3.b32 q1, t, m, o, 0xEA;\n"
        "shr.u32 t, %5, 8;\n lop3.b32 q2, t, m, o, 0xEA;\n"
        "shr.u32 t, %5, 12;\n lop3.b32 q3, t, m, o, 0xEA;\n"
        "sub.rn.bf16x2 p0, p0, k;\n sub.rn.bf16x2 p1, p1, k;\n sub.rn.bf16x2 p2, p2, k;\n sub.rn.bf16x2 p3, p3, k;\n"
        "sub.rn.bf16x2 q0, q0, k;\n sub.rn.bf16x2 q1, q1, k;\n sub.rn.bf16x2 q2, q2, k;\n sub.rn.bf16x2 q3, q3, k;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {p0,q0,p1,q1}, {%6,%7}, {%0,%1,%2,%3};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {p2,q2,p3,q3}, {%8,%9}, {%0,%1,%2,%3};\n"
        "}\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(x2), "r"(x3));
}

// The fp16 form of unpack_mma2_1 (x held in fp16; see unpack_mma2_f16).
__device__ __forceinline__ void unpack_mma2_1_f16(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t x0, uint32_t x1,
                                                  uint32_t x2, uint32_t x3)
{
    asm("{\n"
        ".reg .b32 p0, p1, p2, p3, q0, q1, q2, q3, t, u, ml, mh, o, k, s, b;\n"
        "mov.b32 ml, 0x000F000F;\n"
        "mov.b32 mh, 0x00F000F0;\n"
        "mov.b32 o, 0x64006400;\n"
        "mov.b32 k, 0x64086408;\n"
        "mov.b32 s, 0x2C002C00;\n"
        "mov.b32 b, 0xD480D480;\n"
        "lop3.b32 p0, %4, ml, o, 0xEA;\n"
        "lop3.b32 p1, %4, mh, o, 0xEA;\n"
        "shr.u32 t, %4, 8;\n"
        "lop3.b32 p2, t, ml, o, 0xEA;\n"
        "lop3.b32 p3, t, mh, o, 0xEA;\n"
        "lop3.b32 q0, %5, ml, o, 0xEA;\n"
        "lop3.b32 q1, %5, mh, o, 0xEA;\n"
        "shr.u32 u, %5, 8;\n"
        "lop3.b32 q2, u, ml, o, 0xEA;\n"
        "lop3.b32 q3, u, mh, o, 0xEA;\n"
        "sub.rn.f16x2 p0, p0, k;\n fma.rn.f16x2 p1, p1, s, b;\n sub.rn.f16x2 p2, p2, k;\n fma.rn.f16x2 p3, p3, s, b;\n"
        "sub.rn.f16x2 q0, q0, k;\n fma.rn.f16x2 q1, q1, s, b;\n sub.rn.f16x2 q2, q2, k;\n fma.rn.f16x2 q3, q3, s, b;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {p0,q0,p1,q1}, {%6,%7}, {%0,%1,%2,%3};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {p2,q2,p3,q3}, {%8,%9}, {%0,%1,%2,%3};\n"
        "}\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(x2), "r"(x3));
}

// Two bf16 values (low half first) as two fp16 values, and whether both are
// exact there: zero, or an exponent in [-17, 15] (8 significant bits then fit
// fp16's normal range or its subnormal grid of 2^-24). Other values (larger,
// smaller, bf16 subnormals, inf, NaN) clear ok.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_exact(uint32_t u, bool &ok)
{
    uint32_t r = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t b = (u >> (16 * h)) & 0xFFFFu;
        const uint32_t e = (b >> 7) & 0xFFu;
        ok = ok && ((b & 0x7FFFu) == 0 || (e >= 110u && e <= 142u));
        const __half v = __float2half_rn(__uint_as_float(b << 16));
        r |= (uint32_t)__half_as_ushort(v) << (16 * h);
    }
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Codes `shift` and `shift + 4` of a packed word times the step s, rounded to
// bf16 (nearest even) and packed low-first. (code - 8) * s has at most 12
// significant bits, so the fp32 product is exact and the rounding is the only one.
__device__ __forceinline__ uint32_t bf16x2_of_codes(uint32_t w, int shift, float s)
{
    const float lo = (float)((int)((w >> shift) & 0xFu) - 8) * s;
    const float hi = (float)((int)((w >> (shift + 4)) & 0xFu) - 8) * s;
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&r);
}

// Fused rotation for the Hadamard-rotated GEMV at M = 1 (blocks of b = 32 * PL
// values, PL = 8 or 16, K % 128 == 0; used by the M <= 2 register-preload
// kernel and the shared-memory slot form below vocabulary sizes): xs[0 .. cpr)
// and xs[cpr .. 2 cpr) become the rows hi = bf16(v), lo = bf16(v - hi) of v =
// (x H)[k] (times norm), each 8-value chunk permuted as permute_x8 lays it out.
// Warp w transforms blocks w, w + nwarps, ...: lane l holds values
// [PL*l, PL*l + PL) of the block in registers, so the butterfly stages over
// the low log2(PL) index bits stay in the lane and the next 5 are lane-bit
// exchanges (shfl_xor). Stage order and pairing (p + q, p - q) are those of
// the standalone transform kernel, so both paths give the same bits. All of a
// warp's x loads are issued before its first stage.
template <int PL>
__device__ __forceinline__ void stage_x_hadamard(uint4 *xs, const uint16_t *x, int K, int cpr, float norm)
{
    constexpr int B = 32 * PL, NC = PL / 8; // values and 8-value chunks per lane
    constexpr int kMaxBlk = 1;             // blocks a warp keeps in flight
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int blk0 = threadIdx.x >> 5; blk0 * B < K; blk0 += kMaxBlk * nw) {
        uint4 raw[kMaxBlk][NC];
#pragma unroll
        for (int q = 0; q < kMaxBlk; ++q) {
            const int blk = blk0 + q * nw;
#pragma unroll
            for (int c = 0; c < NC; ++c)
                raw[q][c] = blk * B < K ? *reinterpret_cast<const uint4 *>(x + blk * B + lane * PL + 8 * c)
                                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kMaxBlk; ++q) {
            const int blk = blk0 + q * nw;
            if (blk * B >= K)
                break;
            float v[PL];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t u[4] = {raw[q][c].x, raw[q][c].y, raw[q][c].z, raw[q][c].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * c + 2 * j] = bf16lo_to_f32(u[j]);
                    v[8 * c + 2 * j + 1] = bf16hi_to_f32(u[j]);
                }
            }
#pragma unroll
            for (int h = 1; h < PL; h <<= 1)
#pragma unroll
                for (int r = 0; r < PL; ++r)
                    if (!(r & h)) {
                        const float pv = v[r], qv = v[r + h];
                        v[r] = pv + qv;
                        v[r + h] = pv - qv;
                    }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int r = 0; r < PL; ++r) {
                    const float o = __shfl_xor_sync(0xFFFFFFFFu, v[r], m);
                    v[r] = upper ? o - v[r] : v[r] + o;
                }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float r0 = v[8 * c + 2 * j] * norm, r1 = v[8 * c + 2 * j + 1] * norm;
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(r0), h1 = __float2bfloat16_rn(r1);
                    const __nv_bfloat16 l0 = __float2bfloat16_rn(r0 - __bfloat162float(h0));
                    const __nv_bfloat16 l1 = __float2bfloat16_rn(r1 - __bfloat162float(h1));
                    hw[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                    lw[j] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                const int cc = ((blk * B + lane * PL) >> 3) + c;
                xs[cc] = permute_x8(make_uint4(hw[0], hw[1], hw[2], hw[3]));
                xs[cpr + cc] = permute_x8(make_uint4(lw[0], lw[1], lw[2], lw[3]));
            }
        }
    }
}

// ------------------------------------------------------------- argmax ----

// Order-preserving 64-bit key of (value, index): a larger value wins, and for
// equal values the lower index wins. -0 is folded into +0 first.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx)
{
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u)
        u = 0u;
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long key)
{
    return 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b)
{
    return a > b ? a : b;
}

} // namespace w4
