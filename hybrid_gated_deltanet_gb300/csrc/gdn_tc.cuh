// gdn_tc.cuh -- tcgen05 (5th-generation tensor core) building blocks for
// sm_103a, as inline PTX: TMEM allocation, shared-memory matrix descriptors
// for 128-byte-swizzled K-major TF32 tiles, MMA issue, commit, TMEM loads and
// stores.
//
// Tile convention (K-major, SWIZZLE_128B, TF32 = 4-byte elements): a tile of
// R rows x KW elements (KW a multiple of 32) is stored as KW/32 "atoms" of
// R rows x 128 bytes; element (r, k) sits in atom k/32, row r, 16-byte chunk
// ((k % 32) / 4) XOR (r % 8), position k % 4.  Tiles start on 1024-byte
// boundaries.  One MMA consumes K = 8 (32 bytes of each row); stepping K
// inside an atom advances the descriptor's start address by 32 bytes.
//
// Accumulator layout in TMEM (measured on GB300): for M = 128, row r of D is
// TMEM lane r; for M = 64, row i is lane 32*(i/16) + i%16.  Columns are the
// N index.  A warp may only touch the 32-lane quadrant (warp % 4).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) in a K-major SW128 TF32 tile of `rows` rows
__device__ __forceinline__ uint32_t sw_off(int rows, int r, int k) {
    const int atom = k >> 5, kk = k & 31;
    return (uint32_t)(atom * rows * 128 + r * 128 + ((((kk >> 2) ^ (r & 7))) << 4) + ((kk & 3) << 2));
}

__device__ __forceinline__ float to_tf32_rn(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// store 4 consecutive k of row r (k % 4 == 0), rounded to TF32
__device__ __forceinline__ void st_row4(unsigned char* tile, int rows, int r, int k, float a, float b, float c,
                                        float d) {
    *reinterpret_cast<float4*>(tile + sw_off(rows, r, k)) =
        make_float4(to_tf32_rn(a), to_tf32_rn(b), to_tf32_rn(c), to_tf32_rn(d));
}

__device__ __forceinline__ void st_elem(unsigned char* tile, int rows, int r, int k, float v) {
    *reinterpret_cast<float*>(tile + sw_off(rows, r, k)) = to_tf32_rn(v);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(16 >> 4) << 16;     // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // SWIZZLE_128B
    return d;
}

// instruction descriptor: D f32, A/B tf32, both K-major, M x N
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool negate_a = false) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (negate_a ? (1u << 13) : 0u) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[M x K] * B[N x K]^T over K (multiple of 8), A and B SW128
// K-major TF32 tiles with a_rows / b_rows rows.  Issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, const void* a_tile, int a_rows, const void* b_tile,
                                         int b_rows, int K, uint32_t idesc, bool accumulate) {
    const uint32_t a0 = smem_addr(a_tile), b0 = smem_addr(b_tile);
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint32_t koff = (uint32_t)((k0 & 31) * 4);
        const uint64_t ad = sdesc(a0 + (uint32_t)((k0 >> 5) * a_rows * 128) + koff);
        const uint64_t bd = sdesc(b0 + (uint32_t)((k0 >> 5) * b_rows * 128) + koff);
        const uint32_t acc = (accumulate || k0 > 0) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
            "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
            : "memory");
    }
}

// The K-steps s = part, part + nparts, ... of that product, into accumulator
// d_tmem + part * acc_cols: nparts threads (in different warps) issue the
// parts of one product side by side and the caller adds the nparts partial
// results.  accumulate_first: part 0 adds onto the accumulator's contents,
// the other parts start from zero.
__device__ __forceinline__ void mma_tf32_part(uint32_t d_tmem, const void* a_tile, int a_rows, const void* b_tile,
                                              int b_rows, int K, uint32_t idesc, int part, int nparts, int acc_cols,
                                              bool accumulate_first) {
    const uint32_t a0 = smem_addr(a_tile), b0 = smem_addr(b_tile);
    const uint32_t d = d_tmem + (uint32_t)(part * acc_cols);
    for (int s = part, k0 = part * 8; k0 < K; s += nparts, k0 += 8 * nparts) {
        const uint32_t koff = (uint32_t)((k0 & 31) * 4);
        const uint64_t ad = sdesc(a0 + (uint32_t)((k0 >> 5) * a_rows * 128) + koff);
        const uint64_t bd = sdesc(b0 + (uint32_t)((k0 >> 5) * b_rows * 128) + koff);
        const uint32_t acc = (s >= nparts || (part == 0 && accumulate_first)) ? 1u : 0u;
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
            : "memory");
    }
}

__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 16 consecutive columns of this warp's 32 lanes (thread = lane)
__device__ __forceinline__ void ld16(uint32_t taddr, float v[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// two loads of 16 columns, one wait
__device__ __forceinline__ void ld16x2(uint32_t ta, float va[16], uint32_t tb, float vb[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(ta));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(tb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

// sum of 16 consecutive columns over four accumulators `stride` columns apart
__device__ __forceinline__ void ld16_sum4(uint32_t ta, uint32_t stride, float v[16]) {
    uint32_t r[64];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[16 * q + 0]), "=r"(r[16 * q + 1]), "=r"(r[16 * q + 2]), "=r"(r[16 * q + 3]),
              "=r"(r[16 * q + 4]), "=r"(r[16 * q + 5]), "=r"(r[16 * q + 6]), "=r"(r[16 * q + 7]),
              "=r"(r[16 * q + 8]), "=r"(r[16 * q + 9]), "=r"(r[16 * q + 10]), "=r"(r[16 * q + 11]),
              "=r"(r[16 * q + 12]), "=r"(r[16 * q + 13]), "=r"(r[16 * q + 14]), "=r"(r[16 * q + 15])
            : "r"(ta + q * stride));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = (__uint_as_float(r[i]) + __uint_as_float(r[16 + i])) +
               (__uint_as_float(r[32 + i]) + __uint_as_float(r[48 + i]));
}

__device__ __forceinline__ void st16(uint32_t taddr, const float v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- fp16 operands (kind::f16) -------------------------------------------------
// fp16 tiles use the same 128-byte swizzle: a row of an atom holds 64 fp16
// values (8 chunks of 16 bytes, chunk index XOR row % 8).  One MMA consumes
// K = 16.  K-major operands step K inside an atom by 32 bytes; MN-major
// operands ([K rows][MN], 64 MN values per atom row) step K by 16 rows (2048
// bytes), and the leading byte offset is the stride between 64-wide MN atoms.

// byte offset of the 16-byte chunk cc (elements 8 cc .. 8 cc + 7) of row r of
// an fp16 SW128 atom
__device__ __forceinline__ uint32_t h_off(int r, int cc) {
    return (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t sdesc_lbo(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;  // stride between MN atoms (MN-major operands)
    d |= (uint64_t)(1024 >> 4) << 32;            // next 8-row group
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// instruction descriptor: D f32, A/B fp16, A/B K-major unless *_mn, M x N
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// two floats -> fp16x2 (round to nearest), as a 32-bit word (low half = a)
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 unpack_h2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return __half22float2(h);
}

// 32 consecutive columns of this warp's 32 lanes, no wait
__device__ __forceinline__ void ld32_nowait(uint32_t taddr, uint32_t r[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 64 consecutive columns (two loads, one wait)
__device__ __forceinline__ void ld64(uint32_t taddr, float v[64]) {
    uint32_t r[64];
    ld32_nowait(taddr, r);
    ld32_nowait(taddr + 32, r + 32);
    ld_wait();
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive columns
__device__ __forceinline__ void ld32(uint32_t taddr, float v[32]) {
    uint32_t r[32];
    ld32_nowait(taddr, r);
    ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// store 16 consecutive columns, no wait
__device__ __forceinline__ void st16_nowait(uint32_t taddr, const float v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// TMEM address of (lane, column) relative to an allocation base
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) {
    return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

}  // namespace tc
}  // namespace gdn
