// Blackwell (sm_103a) tensor-core helpers: tcgen05 MMAs with accumulators in tensor memory (TMEM),
// shared-memory matrix descriptors for 128-byte-swizzled operand tiles, TMA tile loads, and
// mbarriers with bounded waits.
//
// Operand tiles (bf16) use the 128-byte swizzle: a tile is a stack of 1024-byte atoms of 8 rows x
// 128 bytes; the 16-byte chunk j of row r is stored at chunk position j ^ (r % 8).  TMA loads with
// CU_TENSOR_MAP_SWIZZLE_128B produce exactly this image, and threads that write tiles apply the
// same XOR.  Two orientations are used:
//   K-major  ([M or N rows][K]):  one 128-byte row = 64 K-values of one row; atoms of 8 rows are
//            SBO bytes apart; a K-step of 16 advances the start address by 32 bytes; a K range
//            beyond 64 lives in a second block of rows.
//   MN-major ([K rows][M or N]):  one 128-byte row = 64 M/N-values of one K index; atoms of 8 K
//            rows are SBO bytes apart; blocks of 64 M/N-values are LBO bytes apart; a K-step of 16
//            advances the start address by two atoms.
// Accumulators: with M = 128 and one CTA, row i of D lives in TMEM lane i, column j in TMEM column
// (base + j), FP32.  Warp w may read lanes 32 (w % 4) .. 32 (w % 4) + 31.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <stdint.h>

#include "kda_mma.cuh"

namespace kda {
namespace tc {

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarriers ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of asynchronous transactions to come.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete; gives up after limit_ns nanoseconds of
// global time and returns false (the caller records an error and stops issuing work).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 1000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// ---- TMA ----
// 2-D tile load into shared memory; completion is counted on `bar` as transaction bytes.
// x (innermost coordinate) must be a multiple of 8 for bf16 data.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// Linear (untiled) copy of `bytes` from global to shared memory by the TMA unit; both addresses
// 16-byte aligned, bytes a multiple of 16; completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// 3-D tiled tensor load into shared memory (coordinates innermost first); completion is counted
// on `bar` as transaction bytes.  x (innermost coordinate) times the element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* map, int x, int y, int z,
                                     uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// 4-D and 5-D tiled tensor loads (one operation fills a whole multi-block operand image).
__device__ __forceinline__ void tma4(void* dst, const CUtensorMap* map, int x, int y, int z, int u,
                                     uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(u), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma5(void* dst, const CUtensorMap* map, int x, int y, int z, int u,
                                     int v, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(u), "r"(v),
        "r"(smem_u32(bar))
        : "memory");
}
// 3-D tiled tensor store from shared memory (the map's swizzle describes the shared image),
// tracked as a bulk async-group of the issuing thread: commit it with bulk_commit, then
// bulk_wait_read0 before the shared tile is rewritten and bulk_wait0 before the block exits.
__device__ __forceinline__ void tma_store3(const CUtensorMap* map, int x, int y, int z,
                                           const void* src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// First 1024-byte boundary at or after p (128-byte-swizzled tiles need it).
__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                            ~uintptr_t(1023));
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (tensor-core operand fetches, TMA stores).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tensor memory ----
// Allocation and release are warp-wide; the allocated base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Loads 32 consecutive FP32 columns of this warp's 32 lanes (thread i gets lane base + i) and
// waits for the load in the same statement, so no use of v can be scheduled before the data.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31])
        : "r"(taddr)
        : "memory");
}

// Stores 32 consecutive FP32 columns of this warp's 32 lanes (thread i writes lane base + i) and
// waits for the store to complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

// ---- MMA ----
// Instruction descriptor of kind::f16 with bf16 A and B, FP32 accumulation; a_mn / b_mn select
// MN-major operand tiles (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor of a 128-byte-swizzled tile starting at saddr (the atom base
// must be 1024-byte aligned; the start may sit 32-byte steps inside an atom's row for K-steps).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A * B, issued by one thread.  acc = 0 overwrites D.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                    uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrives once on `bar` when every MMA issued so far by this thread has completed (including its
// shared-memory operand reads).
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// Abort path of a block whose wait timed out (reached only when the device is already in a bad
// state): one more commit, on a spare barrier initialised here, arrives once every MMA this
// thread issued before it has completed; wait for it (bounded) so that no MMA still writes TMEM
// or reads shared memory when the block frees its TMEM and exits.
__device__ __forceinline__ void drain_mmas(uint64_t* spare, uint64_t limit_ns) {
    mbar_init(spare, 1);
    fence_mbar_init();
    mma_commit(spare);
    mbar_wait(spare, 0, limit_ns);
}

// Writes 32 consecutive values (columns c0..c0+31 of row `row`) of a 128-byte-swizzled bf16 tile
// whose rows hold 64 values, as hi and lo planes; c0 is a multiple of 8.
__device__ __forceinline__ void st_sw128_split32(unsigned char* hi_tile, unsigned char* lo_tile,
                                                 int row, int c0, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2(v[8 * j + 2 * e], v[8 * j + 2 * e + 1], h[e], l[e]);
        const int chunk = ((c0 >> 3) + j) ^ (row & 7);
        const int off = row * 128 + chunk * 16;
        *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// N values (N a multiple of 8) -> packed bf16 hi / lo pairs
template <int N>
__device__ __forceinline__ void split_n(const float (&v)[N], uint32_t (&h)[N / 2], uint32_t (&l)[N / 2]) {
#pragma unroll
    for (int e = 0; e < N / 2; ++e) split2(v[2 * e], v[2 * e + 1], h[e], l[e]);
}
// 128-byte-swizzled tile row `row`: N values (packed pairs) starting at column c0 (multiple of 8)
template <int N>
__device__ __forceinline__ void st_sw128_n(unsigned char* tile, int row, int c0,
                                           const uint32_t (&x)[N / 2]) {
#pragma unroll
    for (int j = 0; j < N / 8; ++j) {
        const int chunk = ((c0 >> 3) + j) ^ (row & 7);
        *reinterpret_cast<uint4*>(tile + row * 128 + chunk * 16) =
            make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
}
// N consecutive bf16 in global memory (16-byte aligned)
template <int N>
__device__ __forceinline__ void st_g_n(__nv_bfloat16* dst, const uint32_t (&x)[N / 2]) {
#pragma unroll
    for (int j = 0; j < N / 8; ++j)
        reinterpret_cast<uint4*>(dst)[j] = make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
}
// Row stores from a warp whose lane i holds row r0 + i (as after a 32x32b tcgen05.ld): the lane
// pairs (2k, 2k + 1) swap 16-byte chunks so that every warp store writes 32 contiguous bytes of
// one row per pair -- whole 32-byte sectors, where one row per lane fills half a sector per
// lane and takes twice the sector writes.  `own` points at this lane's row segment of NC chunks
// (NC even), `ld` is the row stride in 32-bit words; ok0 / ok1 gate the stores of the pair's
// even / odd row.  Every lane of the warp takes part (shuffles).
template <int NC>
__device__ __forceinline__ void st_rows_paired(uint32_t* own, size_t ld, const uint4 (&c)[NC],
                                               int lane, bool ok0, bool ok1) {
    static_assert(NC % 2 == 0, "chunks are exchanged in pairs");
    const bool odd = lane & 1;
    uint32_t* d0 = odd ? own - ld + 4 : own;  // the even row, this lane's chunk of each pair
    uint32_t* d1 = odd ? own + 4 : own + ld;  // the odd row
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) {
        const uint4 ce = c[2 * i], co = c[2 * i + 1];
        const uint4 snd = odd ? ce : co;
        uint4 rcv;
        rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, 1);
        rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, 1);
        rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, 1);
        rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, 1);
        if (ok0) reinterpret_cast<uint4*>(d0 + 8 * i)[0] = odd ? rcv : ce;
        if (ok1) reinterpret_cast<uint4*>(d1 + 8 * i)[0] = odd ? co : rcv;
    }
}
// The same for N consecutive FP32 values of this lane's row (N a multiple of 8).
template <int N>
__device__ __forceinline__ void st_rows_paired_f32(float* own, size_t ld, const float (&v)[N],
                                                   int lane, bool ok0, bool ok1) {
    uint4 c[N / 4];
#pragma unroll
    for (int j = 0; j < N / 4; ++j)
        c[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                          __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
    st_rows_paired<N / 4>(reinterpret_cast<uint32_t*>(own), ld, c, lane, ok0, ok1);
}
// N = 32, 16 or 8 consecutive FP32 TMEM columns of this warp's 32 lanes (as tmem_ld32)
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
    tmem_ld32(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7])
        : "r"(taddr)
        : "memory");
}

// 32 values -> packed bf16 hi / lo pairs
__device__ __forceinline__ void split32(const float (&v)[32], uint32_t (&h)[16],
                                        uint32_t (&l)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) split2(v[2 * e], v[2 * e + 1], h[e], l[e]);
}
// 128-byte-swizzled tile row `row`, 32 values starting at column c0 (multiple of 8)
__device__ __forceinline__ void st_sw128(unsigned char* tile, int row, int c0,
                                         const uint32_t (&x)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int chunk = ((c0 >> 3) + j) ^ (row & 7);
        *reinterpret_cast<uint4*>(tile + row * 128 + chunk * 16) =
            make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
}
// 32 consecutive bf16 in global memory (64 bytes, 16-byte aligned)
__device__ __forceinline__ void st_g32(__nv_bfloat16* dst, const uint32_t (&x)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        reinterpret_cast<uint4*>(dst)[j] = make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
}


}  // namespace tc
}  // namespace kda
