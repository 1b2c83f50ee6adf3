// Warp-level tensor-core helpers: bf16 m16n8k16 MMA with FP32 accumulation, ldmatrix fragment
// loads, the bf16 hi/lo split that makes products FP32-accurate, and cp.async staging.
//
// Split products.  x = hi + lo with hi = bf16(x), lo = bf16(x - hi) keeps ~16 significant bits;
// a * b is taken as a_hi b_hi + a_hi b_lo + a_lo b_hi (three MMAs, relative error ~2^-16), or as
// a_hi b + a_lo b (two MMAs) when b is exactly representable in bf16 (an input such as k, v, dO).
// All partial products accumulate in FP32 in a fixed order, so results are deterministic.
//
// Fragment layout of mma.m16n8k16 (g = lane / 4, t = lane % 4):
//   A (16x16, row): a0a1 (g, 2t..2t+1)  a2a3 (g+8, 2t..)  a4a5 (g, 2t+8..)  a6a7 (g+8, 2t+8..)
//   B (16x8, col):  b0b1 (k = 2t..2t+1, n = g)  b2b3 (k = 2t+8.., n = g)
//   C (16x8):       c0c1 (g, 2t..2t+1)  c2c3 (g+8, 2t..2t+1)
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

namespace kda {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t bits(__nv_bfloat162 v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    return u;
}

// (x0 at the lower column, x1 at the upper) -> packed bf16x2 hi and lo parts
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    hi = bits(h);
    lo = bits(__floats2bfloat162_rn(x0 - hf.x, x1 - hf.y));
}

__device__ __forceinline__ uint32_t pack2(float x0, float x1) {
    return bits(__floats2bfloat162_rn(x0, x1));
}

// Not volatile: a pure register operation, so the compiler may interleave independent MMAs.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// three-term split product into one accumulator: ah*bh + ah*bl + al*bh (small terms first)
__device__ __forceinline__ void mma_x3(float (&d)[4], const uint32_t (&ah)[4],
                                       const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1,
                                       uint32_t bl0, uint32_t bl1) {
    mma16816(d, al, bh0, bh1);
    mma16816(d, ah, bl0, bl1);
    mma16816(d, ah, bh0, bh1);
}

// two-term split product when B is exact in bf16
__device__ __forceinline__ void mma_x2(float (&d)[4], const uint32_t (&ah)[4],
                                       const uint32_t (&al)[4], uint32_t b0, uint32_t b1) {
    mma16816(d, al, b0, b1);
    mma16816(d, ah, b0, b1);
}

// two-term split product when A is exact in bf16
__device__ __forceinline__ void mma_x2b(float (&d)[4], const uint32_t (&a)[4], uint32_t bh0,
                                        uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma16816(d, a, bl0, bl1);
    mma16816(d, a, bh0, bh1);
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// Address of this lane for an A fragment (16x16 at (m0, k0)) of a row-major [m][k] bf16 tile.
__device__ __forceinline__ const __nv_bfloat16* a_addr(const __nv_bfloat16* base, int ld, int m0,
                                                       int k0, int lane) {
    return base + (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ld + k0 + 8 * (lane >> 4);
}
// Same A fragment when the tile is stored transposed, [k][m] (use with ldsm4t).
__device__ __forceinline__ const __nv_bfloat16* at_addr(const __nv_bfloat16* base, int ld, int m0,
                                                        int k0, int lane) {
    return base + (k0 + (lane & 7) + 8 * (lane >> 4)) * ld + m0 + 8 * ((lane >> 3) & 1);
}
// B fragments of two adjacent n-tiles (16(k) x 16(n) at (k0, n0)) of a tile stored [n][k]
// (use with ldsm4): regs {0,1} = n-tile n0, {2,3} = n-tile n0 + 8.
__device__ __forceinline__ const __nv_bfloat16* bn_addr(const __nv_bfloat16* base, int ld, int k0,
                                                        int n0, int lane) {
    return base + (n0 + (lane & 7) + 8 * (lane >> 4)) * ld + k0 + 8 * ((lane >> 3) & 1);
}
// Same when the tile is stored [k][n] (use with ldsm4t).
__device__ __forceinline__ const __nv_bfloat16* bk_addr(const __nv_bfloat16* base, int ld, int k0,
                                                        int n0, int lane) {
    return base + (k0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ld + n0 + 8 * (lane >> 4);
}

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id` (1..15; 0 is the
// block-wide barrier of __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// ---- cp.async (16-byte, L2-cached) ----
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
// 16-byte copy that writes zeros instead when !valid (gmem must still be a valid address)
__device__ __forceinline__ void cp16z(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Copies a [rows][cols] bf16 tile (cols multiple of 8) from a dense global array into a padded
// shared tile with row stride ld, by the whole block.
__device__ __forceinline__ void cp_tile_bf16(__nv_bfloat16* s, int ld, const __nv_bfloat16* g,
                                             int gld, int rows, int cols, int tid, int nthr) {
    const int per_row = cols / 8;
    for (int i = tid; i < rows * per_row; i += nthr) {
        const int r = i / per_row, c = (i % per_row) * 8;
        cp16(s + r * ld + c, g + size_t(r) * gld + c);
    }
}
// Same for fp32 tiles (cols multiple of 4).
__device__ __forceinline__ void cp_tile_f32(float* s, int ld, const float* g, int gld, int rows,
                                            int cols, int tid, int nthr) {
    const int per_row = cols / 4;
    for (int i = tid; i < rows * per_row; i += nthr) {
        const int r = i / per_row, c = (i % per_row) * 4;
        cp16(s + r * ld + c, g + size_t(r) * gld + c);
    }
}

// Copies a [rows][cols] bf16 shared tile (row stride sld) to a dense global tile (row stride gld)
// with 16-byte accesses by the whole block; flip = 0x80008000 negates every element.
__device__ __forceinline__ void st_tile_bf16(__nv_bfloat16* g, int gld, const __nv_bfloat16* s,
                                             int sld, int rows, int cols, int tid, int nthr,
                                             uint32_t flip = 0u) {
    const int per_row = cols / 8;
    for (int i = tid; i < rows * per_row; i += nthr) {
        const int r = i / per_row, c = (i % per_row) * 8;
        uint4 v = *reinterpret_cast<const uint4*>(s + r * sld + c);
        v.x ^= flip;
        v.y ^= flip;
        v.z ^= flip;
        v.w ^= flip;
        *reinterpret_cast<uint4*>(g + size_t(r) * gld + c) = v;
    }
}

}  // namespace kda
