// kda_tc.cuh -- inline-PTX helpers for the 5th-generation tensor cores (tcgen05) on sm_100+:
// tensor-memory allocation, shared-memory matrix descriptors, MMA issue / commit, TMEM loads,
// and the bf16 "split" staging that carries FP32 operands through bf16 MMAs.
//
// Operand layout used throughout: a [R x Kt] bf16 tile, K-major, no swizzle, stored as 8 x 8
// "core matrices" (8 rows x 16 bytes, 128 contiguous bytes each).  With the 16-byte chunks
// enumerated q = rg * (8 * Kt/8) + kg * 8 + (r % 8)   (rg = r / 8, kg = k / 8), chunk q lives at
// byte q * 16: core matrices adjacent in K are 128 bytes apart (leading byte offset) and 8-row
// groups Kt * 16 bytes apart (stride byte offset).  One MMA consumes K = 16, i.e. two core
// matrices along K, so the k-th step starts 256 bytes further.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_ptx.cuh"

namespace kda {
namespace tc {

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version for sm_100 family; no swizzle, base offset 0
    return d;
}

// Instruction descriptor: kind::f16, A and B bf16, K-major, D f32, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of element (r, k) in a core-matrix tile with Kt columns.
__host__ __device__ constexpr uint32_t cm_off(int r, int k, int Kt)
{
    return (uint32_t)((r >> 3) * (Kt >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// 16-byte chunk q of a tile with Kt columns -> (row, first k).
__device__ __forceinline__ void cm_chunk(int q, int Kt, int &r, int &k)
{
    const int per_rg = Kt;   // 8 rows x Kt/8 chunks
    const int rg = q / per_rg, rem = q % per_rg;
    r = rg * 8 + (rem & 7);
    k = (rem >> 3) * 8;
}

// Warp-wide TMEM allocation (one warp calls it); the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// D[M=128 x N] (+)= A[128 x K] * B[N x K]^T over K = 16 * ksteps, A and B core-matrix tiles
// with Ka / Kb total columns (their stride byte offsets), starting at k-step k0.
// The descriptors are built once: the next k-step starts 256 bytes further, i.e. 16 more in
// the descriptor's 16-byte-granular address field (shared addresses stay below 256 KiB, so the
// 14-bit field never carries into the next one).
__device__ __forceinline__ void mma_tiles(uint32_t d_tmem, uint32_t a_saddr, int Ka, uint32_t b_saddr, int Kb,
                                          int N, int k0, int ksteps, bool accumulate)
{
    const uint32_t id = idesc_bf16(128, N);
    uint64_t ad = smem_desc(a_saddr + (uint32_t)k0 * 256u, 128u, (uint32_t)Ka * 16u);
    uint64_t bd = smem_desc(b_saddr + (uint32_t)k0 * 256u, 128u, (uint32_t)Kb * 16u);
#pragma unroll
    for (int s = 0; s < ksteps; s++) {
        mma(d_tmem, ad, bd, id, accumulate || s > 0);
        ad += 16u;
        bd += 16u;
    }
}

// FP32-accurate product from bf16 MMAs: D (+)= Ah Bh^T + Ah Bl^T + Al Bh^T, where X = Xh + Xl
// with Xh = bf16(X) and Xl = bf16(X - Xh) (about 16 significant bits per operand).
__device__ __forceinline__ void mma_split3(uint32_t d_tmem, uint32_t ah, uint32_t al, int Ka, uint32_t bh,
                                           uint32_t bl, int Kb, int N, int ksteps, bool accumulate)
{
    mma_tiles(d_tmem, ah, Ka, bh, Kb, N, 0, ksteps, accumulate);
    mma_tiles(d_tmem, ah, Ka, bl, Kb, N, 0, ksteps, true);
    mma_tiles(d_tmem, al, Ka, bh, Kb, N, 0, ksteps, true);
}

// The same split product with a K-major B stored as [Bh ; Bl] (2N rows, Bl right after Bh): Ah
// against both halves at once (N' = 2N), then Al Bh^T onto the first N columns.  The product is
// D[0, N) + D[N, 2N): two A passes instead of three.
__device__ __forceinline__ void mma_split3_kcat(uint32_t d_tmem, uint32_t ah, uint32_t al, int Ka, uint32_t bcat,
                                                int Kb, int N, int ksteps, bool accumulate)
{
    mma_tiles(d_tmem, ah, Ka, bcat, Kb, 2 * N, 0, ksteps, accumulate);
    mma_tiles(d_tmem, al, Ka, bcat, Kb, N, 0, ksteps, true);
}

// B operands stored MN-major (N contiguous), no swizzle: the core matrix of n-group g and k-group
// q is 8 k-rows of 16 bytes (8 consecutive n) at byte g * 128 + q * (N / 8) * 128, so a thread
// that holds one k-row of B writes it as N / 8 chunks of 16 bytes.  In the shared-memory
// descriptor the leading byte offset is then the step between k-groups and the stride byte offset
// the step between n-groups (measured on GB300 with a single product against a CPU reference);
// bit 16 of the instruction descriptor marks B as MN-major.
__host__ __device__ constexpr uint32_t bmn_off(int n, int k, int N)
{
    return (uint32_t)((n >> 3) * 128 + (k >> 3) * (N >> 3) * 128 + (k & 7) * 16 + (n & 7) * 2);
}

// D[M=128 x N] (+)= A[128 x K] * B[N x K]^T over K = 16 * ksteps: A a K-major core-matrix tile
// with Ka total columns, B MN-major as above with k-groups `kgs` bytes apart (N / 8 x 128 for a
// tile of exactly N columns; more when B is the first N columns of a wider tile).
__device__ __forceinline__ void mma_tiles_bmn_ks(uint32_t d_tmem, uint32_t a_saddr, int Ka, uint32_t b_saddr,
                                                 int N, uint32_t kgs, int ksteps, bool accumulate)
{
    const uint32_t id = idesc_bf16(128, N) | (1u << 16);
    uint64_t ad = smem_desc(a_saddr, 128u, (uint32_t)Ka * 16u);
    uint64_t bd = smem_desc(b_saddr, kgs, 128u);
#pragma unroll
    for (int s = 0; s < ksteps; s++) {
        mma(d_tmem, ad, bd, id, accumulate || s > 0);
        ad += 16u;
        bd += (2u * kgs) >> 4;   // one MMA consumes two k-groups
    }
}

// The same split product with B given as one MN-major tile of 2N columns, [Bh | Bl]: the first
// pass takes Ah against both halves at once (N' = 2N), the second adds Al Bh^T onto the first N
// columns.  The product is D[0, N) + D[N, 2N): two A passes instead of three, so a third less of
// the A operand is read from shared memory.
__device__ __forceinline__ void mma_split3_bcat(uint32_t d_tmem, uint32_t ah, uint32_t al, int Ka, uint32_t bcat,
                                                int N, int ksteps, bool accumulate)
{
    const uint32_t kgs = (uint32_t)(2 * N >> 3) * 128u;
    mma_tiles_bmn_ks(d_tmem, ah, Ka, bcat, 2 * N, kgs, ksteps, accumulate);
    mma_tiles_bmn_ks(d_tmem, al, Ka, bcat, N, kgs, ksteps, true);
}

// Packed FP32 arithmetic: two lanes per instruction, each lane an IEEE round-to-nearest
// operation, so every result equals the scalar form bit for bit.
//   fma2: d = a * b + c        mul2: d = a * b
//   add2: d = a + b (as a * 1 + b: the product is exact, one rounding)
//   sub2: d = a - b (as b * -1 + a)
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    fma2(d0, d1, a0, a1, 1.0f, 1.0f, b0, b1);
}
__device__ __forceinline__ void sub2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    fma2(d0, d1, b0, b1, -1.0f, -1.0f, a0, a1);
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b)
{
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Two floats rounded to bf16 (nearest even) in one conversion, a in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Split 8 consecutive floats into one 16-byte chunk of hi and one of lo: hi = bf16(x),
// lo = bf16(x - hi), with x ~= hi + lo.  x - hi is exact in FP32, so the packed subtraction
// gives the same lo as a scalar one.
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        h[e] = bf16x2_rn(x[2 * e], x[2 * e + 1]);
        float r0, r1;
        sub2(r0, r1, x[2 * e], x[2 * e + 1], __uint_as_float(h[e] << 16), __uint_as_float(h[e] & 0xffff0000u));
        l[e] = bf16x2_rn(r0, r1);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// TMEM -> registers: this warp's 32 lanes (lane quarter warp % 4), 32 consecutive columns.
__device__ __forceinline__ void ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
}

// TMEM -> registers: this warp's 32 lanes, 16 consecutive columns.
__device__ __forceinline__ void ld16(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; j++) v[j] = __uint_as_float(r[j]);
}

// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) { return base + ((uint32_t)lane << 16) + (uint32_t)col; }

}  // namespace tc
}  // namespace kda
