// Per-chunk gradient products of the backward on tcgen05 tensor cores (TMEM accumulators,
// TMA-fed operands), per (chunk, head) item of a persistent block:
//   MMA1  DR  = Minv^T dDelta                      M = 128 (rows 0..63), N = 128 values, K = 64
//   MMA2  DPQ = [dR; dO] S0^T                      rows 0..63: P, rows 64..127: dQg / scale
//   MMA3  DAM = [dR; dO] Delta^T                   rows 0..63: -dM, rows 64..127: dAqk / scale
//   MMA4  DKb = [Delta; *] dS1^T                   rows 0..63: dKb
// and rowsum(S0 * dS1) per key from the two shared tiles (two partials, one per K block).
// dR (rows 0..63 of the [dR; dO] operand) comes from MMA1 through TMEM -> registers -> shared
// memory; dO (rows 64..127) arrives by TMA, its lo plane stays zero.  Every product is a split
// bf16 product (hi/lo planes, three MMAs; FP32 accumulation in TMEM).  Rows 64..127 of the MMA1
// and MMA4 A operands are whatever follows the operand tile in shared memory: they only reach
// accumulator rows that are never read.  dO rows past the chunk's end (the next document's
// tokens, or zeros past T) only reach gradient rows that meet zero-padded q, k, beta later.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

// shared-memory image, byte offsets from a 1024-byte aligned base; plane 0 = hi, 1 = lo
constexpr int G_MN = 0;          // Minv as MN-major A of Minv^T: [plane][64 t][128 B]         16 KB
constexpr int G_DD = 16384;      // dDelta MN-major B: [plane][2 value blocks][64 t][128 B]    32 KB
constexpr int G_A = 49152;       // [dR; dO] K-major A: [plane][2 K blocks][128 rows][128 B]   64 KB
constexpr int G_S0 = 114688;     // S0 K-major B: [plane][2 K blocks][128 keys][128 B]         64 KB
constexpr int G_DL = 180224;     // Delta K-major: [plane][2 K blocks][64 t][128 B]            32 KB
constexpr int G_X = 212992;      // 16 KB: the fourth dS1 tile (the others reuse G_MN / G_DD)
constexpr int G_BAR = 229376;    // mbarriers, TMEM base address
constexpr size_t BWD_GEMM_TC_SMEM = G_BAR + 128 + 1024;

static_assert(BWD_GEMM_TC_SMEM <= 232448, "tcgen05 backward GEMM shared memory above the limit");

// dS1 K-major B tiles [128 keys][128 B] (plane, K block): in the Minv / dDelta space after MMA1
__host__ __device__ constexpr int ds1_tile(int pl, int kb) {
    return pl == 0 ? 16384 * kb : (kb == 0 ? 32768 : G_X);
}

}  // namespace

size_t bwd_gemm_tc_smem_bytes() { return BWD_GEMM_TC_SMEM; }

// Persistent: one block per SM walks the (chunk, head) items item = chunk * H + head.  As soon as
// an item's MMAs and row sums are done, every operand tile is free and the next item's TMA loads
// start, overlapping this item's TMEM -> global epilogues.
__global__ void __launch_bounds__(NTHR, 1) k_bwd_gemms_tc(Params p, const __grid_constant__ TcMaps tm) {
    // no work after a failed device-side check of this call (the outputs stay unwritten)
    const int items = *p.status == KDA_ERR_DEVICE_CHECK ? 0 : *p.nchunks * p.H;
    if (int(blockIdx.x) >= items) return;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = tc::align1024(smraw);
    // 0 G1 in, 1 G2 in, 2 MMA1, 3 MMA2/3, 4 dS1 in, 5 MMA4 (+80: spare barrier of the abort path)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + G_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + G_BAR + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + G_BAR + 68);
    // leave-the-loop decision: thread 0 copies the abort flag into the item's slot (parity) before
    // the barrier and every thread reads that slot after it, so all warps leave together
    volatile int* stopf = reinterpret_cast<volatile int*>(sm + G_BAR + 72);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int qd = w & 3, half = w >> 2;
    const int row = 32 * qd + lane;  // accumulator row / TMEM lane of this thread

    // G1: Minv (hi, lo) and dDelta (hi, lo); G2: dO into rows 64..127 of the hi [dR; dO] operand,
    // S0 and Delta (thread 0; t0 = the item's first token)
    auto issue_loads = [&](int chd, int hh, int t0) {
        tc::mbar_expect_tx(&bar[0], 49152u);
        tc::tma4(sm + G_MN, &tm.mAq, 0, 0, 0, tm.zMh + chd, &bar[0]);         // Minv, both planes
        tc::tma5(sm + G_DD, &tm.mDD5, 0, 0, 0, 0, chd, &bar[0]);              // dDelta, both planes
        tc::mbar_expect_tx(&bar[1], 114688u);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) tc::tma3(sm + G_A + 16384 * kb + 8192, &tm.mdO, 64 * kb, hh, t0, &bar[1]);
        tc::tma5(sm + G_S0, &tm.mS5, 0, 0, 0, 0, chd, &bar[1]);               // S0, both planes
        tc::tma5(sm + G_DL, &tm.mDl5, 0, 0, 0, 0, chd, &bar[1]);              // Delta, both planes
    };
    int pend = -1;  // phase parity of the G1 / G2 loads in flight (thread 0), -1 = none
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 6; ++i) tc::mbar_init(&bar[i], 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        const int first = blockIdx.x;
        issue_loads(first, first % p.H, p.chunk_tab[first / p.H].y);
        pend = 0;
    }
    if (w == 0) tc::tmem_alloc(tslot, 512);
    // lo plane of the dO rows: zero for good (nothing else writes there)
    for (int i = tid; i < 2 * 8192 / 16; i += NTHR) {
        const int kb = i / 512, o = (i % 512) * 16;
        *reinterpret_cast<uint4*>(sm + G_A + 32768 + 16384 * kb + 8192 + o) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tslot;
    const uint32_t tl = taddr + (uint32_t(32 * qd) << 16);
    const int tpa[3] = {0, 1, 0}, tpb[3] = {1, 0, 0};  // (A plane, B plane) of the split terms

    int it = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t ph = uint32_t(it) & 1u;
        const int chd = item;  // chunk * H + head
        const int next = item + int(gridDim.x);
        int t0n = 0, hn = 0;
        if (tid == 0 && next < items) {  // the next item's first token, read early
            t0n = p.chunk_tab[next / p.H].y;
            hn = next % p.H;
        }

        // ---- MMA1: DR = Minv^T dDelta ----
        if (tid == 0) {
            if (tc::mbar_wait(&bar[0], ph)) {
                tc::fence_after_sync();
                const uint32_t sMN = smem_u32(sm + G_MN), sDD = smem_u32(sm + G_DD);
                const uint64_t mh = tc::sdesc(sMN, 8192, 1024), ml = tc::sdesc(sMN + 8192, 8192, 1024);
                const uint64_t dh = tc::sdesc(sDD, 8192, 1024), dl = tc::sdesc(sDD + 16384, 8192, 1024);
                const uint64_t ta[3] = {mh, ml, mh}, tb[3] = {dl, dh, dh};
                const uint32_t id = tc::idesc_bf16(128, 128, true, true);
                uint32_t acc = 0;
#pragma unroll
                for (int t3 = 0; t3 < 3; ++t3)
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        tc::mma(taddr, ta[t3] + uint64_t((s * 2048) >> 4), tb[t3] + uint64_t((s * 2048) >> 4), id, acc);
                        acc = 1;
                    }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[2]);
        }
        __syncwarp();
        if (!tc::mbar_wait(&bar[2], ph)) *abort_flag = 1;
        tc::fence_after_sync();
        if (tid == 0) {  // G3: dS1 into the Minv / dDelta space, free now
            tc::mbar_expect_tx(&bar[4], 65536u);
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                    tc::tma3(sm + ds1_tile(pl, kb), &tm.mdS, 64 * kb, 0, 2 * chd + pl, &bar[4]);
        }
        __syncwarp();

        // ---- dR: fp32 to global, hi / lo split into rows 0..63 of the [dR; dO] operand ----
        if (qd < 2) {
            float* dst = p.dR + size_t(chd) * CH * D + size_t(row) * D + 64 * half;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float v[32];
                tc::tmem_ld32(tl + 64 * half + 32 * q2, v);
                tc::st_rows_paired_f32<32>(dst + 32 * q2, D, v, lane, true, true);
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // 16-byte chunk 4 q2 + j of this row's K-block row
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) split2(v[8 * j + 2 * e], v[8 * j + 2 * e + 1], hi[e], lo[e]);
                    const int off = row * 128 + (((4 * q2 + j) ^ (row & 7)) * 16);
                    *reinterpret_cast<uint4*>(sm + G_A + 16384 * half + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(sm + G_A + 32768 + 16384 * half + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        if (tid == 0) stopf[it & 1] = *abort_flag;
        __syncthreads();
        tc::fence_after_sync();
        if (stopf[it & 1]) break;

        // ---- MMA2 / MMA3 ([dR; dO] S0^T, [dR; dO] Delta^T), then MMA4 (Delta dS1^T) ----
        if (tid == 0) {
            const uint32_t sA = smem_u32(sm + G_A), sS = smem_u32(sm + G_S0), sL = smem_u32(sm + G_DL);
            if (tc::mbar_wait(&bar[1], ph)) {
                pend = -1;
                tc::fence_after_sync();
                const uint32_t i2 = tc::idesc_bf16(128, 128, false, false);
                const uint32_t i3 = tc::idesc_bf16(128, 64, false, false);
                uint32_t acc = 0;
#pragma unroll
                for (int t3 = 0; t3 < 3; ++t3)
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const int kb = s >> 2, ko = (s & 3) * 32;
                        const uint64_t a = tc::sdesc(sA + 32768 * tpa[t3] + 16384 * kb + ko, 16, 1024);
                        const uint64_t b2 = tc::sdesc(sS + 32768 * tpb[t3] + 16384 * kb + ko, 16, 1024);
                        const uint64_t b3 = tc::sdesc(sL + 16384 * tpb[t3] + 8192 * kb + ko, 16, 1024);
                        tc::mma(taddr + 128, a, b2, i2, acc);
                        tc::mma(taddr + 256, a, b3, i3, acc);
                        acc = 1;
                    }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[3]);
            if (tc::mbar_wait(&bar[4], ph)) {
                tc::fence_after_sync();
                const uint32_t i4 = tc::idesc_bf16(128, 128, false, false);
                uint32_t acc = 0;
#pragma unroll
                for (int t3 = 0; t3 < 3; ++t3)
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const int kb = s >> 2, ko = (s & 3) * 32;
                        const uint64_t a = tc::sdesc(sL + 16384 * tpa[t3] + 8192 * kb + ko, 16, 1024);
                        const uint64_t b = tc::sdesc(smem_u32(sm + ds1_tile(tpb[t3], kb)) + ko, 16, 1024);
                        tc::mma(taddr + 320, a, b, i4, acc);
                        acc = 1;
                    }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[5]);
        }
        __syncwarp();

        // ---- rowsum(S0 * dS1) of this thread's key over K block `half` (hi + lo of both) ----
        bool ok = tc::mbar_wait(&bar[4], ph);  // makes the dS1 tiles visible to this thread
        ok = tc::mbar_wait(&bar[3], ph) && ok;
        ok = tc::mbar_wait(&bar[5], ph) && ok;  // every MMA of the item done: all tiles free after
        if (!ok) *abort_flag = 1;
        tc::fence_after_sync();
        {
            const unsigned char* s0h = sm + G_S0 + 16384 * half;
            const unsigned char* d1h = sm + ds1_tile(0, half);
            const unsigned char* d1l = sm + ds1_tile(1, half);
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunks in logical order
                const int off = row * 128 + ((j ^ (row & 7)) * 16);
                const uint4 a = *reinterpret_cast<const uint4*>(s0h + off);
                const uint4 b = *reinterpret_cast<const uint4*>(s0h + 32768 + off);
                const uint4 c = *reinterpret_cast<const uint4*>(d1h + off);
                const uint4 d = *reinterpret_cast<const uint4*>(d1l + off);
                const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
                const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
                const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c);
                const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 s0 = __bfloat1622float2(a2[e]), s1 = __bfloat1622float2(b2[e]);
                    const float2 g0 = __bfloat1622float2(c2[e]), g1 = __bfloat1622float2(d2[e]);
                    part = fmaf(s0.x + s1.x, g0.x + g1.x, part);
                    part = fmaf(s0.y + s1.y, g0.y + g1.y, part);
                }
            }
            p.rsum[(size_t(chd) * 2 + half) * D + row] = part;
        }
        __syncthreads();  // every operand tile is free: the next item's loads start now
        if (tid == 0 && next < items && !*abort_flag) {
            issue_loads(next, hn, t0n);
            pend = int(ph ^ 1u);
        }

        // ---- epilogues from TMEM (overlap the next item's loads) ----
        {
            const bool top = qd < 2;  // lanes 0..63: P and dM rows; lanes 64..127: dQg and dAqk rows
            const int r = top ? row : row - 64;
            float* dst = (top ? p.P : p.dQg) + size_t(chd) * CH * D + size_t(r) * D + 64 * half;
            const float sc = top ? 1.f : p.scale;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float v[32];
                tc::tmem_ld32(tl + 128 + 64 * half + 32 * q2, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= sc;
                tc::st_rows_paired_f32<32>(dst + 32 * q2, D, v, lane, true, true);
            }
            float v[32];
            tc::tmem_ld32(tl + 256 + 32 * half, v);
            float* da = (top ? p.dM : p.dAqk) + size_t(chd) * CH * CH + size_t(r) * CH + 32 * half;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int s = 32 * half + j;
                v[j] = top ? (s < r ? -v[j] : 0.f) : (s <= r ? p.scale * v[j] : 0.f);
            }
            tc::st_rows_paired_f32<32>(da, CH, v, lane, true, true);
        }
        if (qd < 2) {
            float* dst = p.dKb + size_t(chd) * CH * D + size_t(row) * D + 64 * half;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float v[32];
                tc::tmem_ld32(tl + 320 + 64 * half + 32 * q2, v);
                tc::st_rows_paired_f32<32>(dst + 32 * q2, D, v, lane, true, true);
            }
        }
        tc::fence_before_sync();  // TMEM reads above come before the next item's MMAs
    }

    if (*abort_flag && tid == 0) {
        // after a timed-out wait: let this block's MMAs and TMA loads in flight finish (bounded),
        // report
        tc::drain_mmas(reinterpret_cast<uint64_t*>(sm + G_BAR + 80), 100000000ull);
        if (pend >= 0) {
            tc::mbar_wait(&bar[0], uint32_t(pend), 100000000ull);
            tc::mbar_wait(&bar[1], uint32_t(pend), 100000000ull);
        }
        p.status[0] = KDA_ERR_TIMEOUT;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(taddr, 512);
}

}  // namespace kda
