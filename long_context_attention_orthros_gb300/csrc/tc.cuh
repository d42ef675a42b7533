// tc.cuh -- tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor
// memory allocation, shared-memory matrix descriptors, instruction descriptors,
// MMA issue / commit, and tensor-memory loads and stores.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace orthros {

// Shared-memory matrix descriptor, 128-byte swizzle.  For K-major operands the
// 8-row groups are `sbo` bytes apart (lbo unused); for MN-major operands `lbo`
// is the distance between 64-element MN slabs and `sbo` between 8-row K groups.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation; A and B are both
// bf16 (bf16 = true) or both fp16.  B is K-major unless b_mn_major.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, bool bf16, bool b_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]  (issued by one thread)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]  (issued by one thread)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's lane (its warp's quarter of the 128 lanes).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// ------------------------------------------------------------------ keys as fp16 MMA operands
// The tensor-memory kernels take q . k in fp16.  A bf16 key converts to fp16 exactly while
// |k| < 65520 (fp16's range; bf16 values below fp16's normal range keep their value to within
// 2^-25).  A key row whose largest |k| reaches 65520 is scaled by an exact power of two 2^-e
// that puts its largest element in [2^14, 2^15), and its logits are multiplied back by 2^e in
// fp32, so every finite bf16 key is taken.

// 2^n for an integer n in [-126, 127], exactly
__device__ __forceinline__ float exp2i(int n) { return __uint_as_float(static_cast<uint32_t>(127 + n) << 23); }

// largest |x| of eight bf16 values (a NaN is passed over)
__device__ __forceinline__ float bf16x8_absmax(uint4 u)
{
    const uint32_t w[4] = {u.x & 0x7fff7fffu, u.y & 0x7fff7fffu, u.z & 0x7fff7fffu, u.w & 0x7fff7fffu};
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        m = fmax3(m, f.x, f.y);
    }
    return m;
}

// shift e of a key row whose largest |k| is amax: 0 below 65520, else amax * 2^-e lies in
// [2^14, 2^15); an infinite key sets bad (its logits cannot be finite) and keeps e = 0
__device__ __forceinline__ int fp16_key_shift(float amax, bool &bad)
{
    if (amax < 65520.f)
        return 0;
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
    if (ex == 255) {
        bad = true;
        return 0;
    }
    return ex - 127 - 14;
}

// eight bf16 values as fp16 (round to nearest even)
__device__ __forceinline__ uint4 k_to_fp16(uint4 u)
{
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        __half2 hv = __floats2half2_rn(f.x, f.y);
        w[e] = *reinterpret_cast<uint32_t *>(&hv);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// the same after multiplying by sd (a power of two)
__device__ __forceinline__ uint4 k_to_fp16_scaled(uint4 u, float sd)
{
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        __half2 hv = __floats2half2_rn(f.x * sd, f.y * sd);
        w[e] = *reinterpret_cast<uint32_t *>(&hv);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The rare path of a key-block conversion done by one warp, 8 lanes per key row, when one of
// its rows holds a value at or beyond 65520: this lane holds chunk c8 of every slab of rows
// rsub + rstep * r (r < nrows), all still bf16.  Each row's largest |k| over its 8 lanes decides
// its shift e; the row is written as fp16 of k * 2^-e (at blk + sl * slab_bytes, and again
// `mirror` bytes further when mirror != 0) and e is stored at kexp[row].  Called by the whole
// warp.
template <int SLABS>
__device__ __noinline__ void shift_key_rows(uint8_t *blk, int slab_bytes, int mirror, int rsub, int rstep, int nrows,
                                            int c8, int8_t *kexp, bool &bad)
{
#pragma unroll 1
    for (int r = 0; r < nrows; ++r) {
        const int row = rsub + rstep * r;
        float amax = 0.f;
        uint4 u[SLABS];
#pragma unroll
        for (int sl = 0; sl < SLABS; ++sl) {
            u[sl] = *reinterpret_cast<const uint4 *>(blk + sl * slab_bytes + row * 128 + c8 * 16);
            amax = fmaxf(amax, bf16x8_absmax(u[sl]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const int ex = fp16_key_shift(amax, bad);
        if (c8 == 0)
            kexp[row] = static_cast<int8_t>(ex);
        const float sd = exp2i(-ex);
#pragma unroll
        for (int sl = 0; sl < SLABS; ++sl) {
            const uint4 h = k_to_fp16_scaled(u[sl], sd);
            uint8_t *dst = blk + sl * slab_bytes + row * 128 + c8 * 16;
            *reinterpret_cast<uint4 *>(dst) = h;
            if (mirror != 0)
                *reinterpret_cast<uint4 *>(dst + mirror) = h;
        }
    }
}

// The rare path of the softmax warps: the logits of 32 consecutive keys (one 32-column chunk of
// this warp's 32 tensor-memory lanes at taddr; key rows row0 .. row0 + 31 of their block) times
// 2^e_j, read back and stored in place.  Row r's shift is ke[r] when bit ((r % period) / per) of
// wmask is set (the converter warp owning the row found it beyond fp16), else 0.  A logit that is
// no longer finite sets bad.  Called by the whole warp; the caller reloads the chunk afterwards.
static __device__ __noinline__ void unshift_chunk32(uint32_t taddr, const int8_t *ke, int row0, uint32_t wmask, int period,
                                             int per, bool &bad)
{
    uint32_t v[32];
    tmem_ld32(taddr, v);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int r = row0 + e;
        const int x = ((wmask >> ((r % period) / per)) & 1u) ? ke[r] : 0;
        if (x != 0) {
            const float y = __uint_as_float(v[e]) * exp2i(x);
            bad |= isinf(y);
            v[e] = __float_as_uint(y);
        }
    }
    tmem_st32(taddr, v);
    tmem_wait_st();
}

}  // namespace orthros
