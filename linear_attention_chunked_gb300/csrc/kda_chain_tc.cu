// Inter-chunk state recurrence of the forward pass on tcgen05 tensor cores (TMEM accumulators,
// TMA-fed operands).  Per (document, head, block of VW value columns) and chunk, with the FP32
// state S held in registers (thread = one key row x VW / 2 value columns; VW = 16, 32 or 64):
//   MMA1  D1 = [W; Qg] S                 M = 128 (64 W rows, 64 Qg rows), N = VW, K = 128 keys
//         Delta = U - D1[0:64]           (threads of TMEM lanes 0..63)
//   MMA2  D2 = Kb^T Delta                M = 128 keys, N = VW, K = 64 tokens
//   MMA3  D1 += [*; Aqk] Delta           rows 64..127: O = Qg S + Aqk Delta
//         S  = e^gL * S + D2             (every thread, its own row)
// Every product is split into bf16 hi/lo terms (a_hi b_lo + a_lo b_hi + a_hi b_hi, FP32
// accumulate in TMEM), which keeps ~16 significant bits per operand.  The B operand's hi and lo
// planes sit side by side along N (64-column blocks: two 64-column atoms, the lo plane one plane
// stride away; narrower blocks: the lo values at column VW of the hi tile): one N = 2 VW MMA gives
// a_hi b_hi and a_hi b_lo in two TMEM column halves, a_lo b_hi adds onto the first, and the
// epilogues sum the halves -- two MMAs per K step instead of three, A read twice instead of three
// times, and the same arithmetic for every block width (bitwise equal results).  Rows 0..63 of
// the MMA3 A operand are whatever precedes the hi / lo Aqk tiles (zeros / the hi tile): they only
// touch D1 rows whose W S values were already consumed.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

// Shared-memory image, byte offsets from a 1024-byte aligned base.  Operand tiles are 128-byte
// swizzled (see kda_tc.cuh); "plane" 0 = hi, 1 = lo.
constexpr int OFF_KT = 0;        // Kb as MN-major A: [plane][2 key blocks][64 tokens][128 B]  32 KB
constexpr int OFF_A1 = 32768;    // [W; Qg] K-major: [plane][2 key blocks][128 rows][128 B]    64 KB
constexpr int OFF_S = 98304;     // S as MN-major B: [plane][128 keys][128 B] (VW < 64: one plane) 32 KB
constexpr int OFF_PAD = 131072;  // 8 KB of zeros: rows 0..63 of the hi MMA3 operand
constexpr int OFF_AQ = 139264;   // Aqk K-major: [plane][64 tokens][128 B]                     16 KB
constexpr int OFF_DL = 155648;   // Delta as MN-major B: [plane][64 tokens][128 B] (likewise)  16 KB
constexpr int OFF_BAR = 172032;  // mbarriers, TMEM base address, abort flag
constexpr size_t CHAIN_TC_SMEM = OFF_BAR + 128 + 1024;  // + alignment slack of the base

static_assert(CHAIN_TC_SMEM <= 232448, "tcgen05 chain shared memory above the opt-in limit");

}  // namespace


// Grid N x H x (128 / VW) value parts of VW = 64, 32 or 16 columns for CHAIN_FWD_OUT; N x H x 4 parts
// for CHAIN_FRAG_MB (VW = 64; parts 0, 1: X = I with zero values -> M; parts 2, 3: Y = 0 with the
// values -> B).  256 threads: warp w reads TMEM lanes 32 (w % 4).. and VW / 2 value columns from
// VW / 2 (w / 4) of its part.  The per-chunk latency scales with VW, so runs with few (document,
// head) pairs use VW = 16 or 32 (more blocks on the critical path), the others VW = 64.
// Thread 0 issues the MMAs and the TMA stores; thread 96 (warp 3: no Delta rows, and its O rows
// cost more than a TMA issue) issues the TMA loads, so their issue cost stays off thread 0.
// Operands of chunk c+1 are loaded as soon as the MMA that reads their buffer has completed.
template <int VW>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    k_chain_fwd_tc(Params p, int mode, const __grid_constant__ TcMaps tm) {
    constexpr int VPT = VW / 2;  // value columns per thread
    // block = (document rank, head, value part): longest documents first, the parts of one
    // (document, head) adjacent so their shared operand tiles are read from L2 together
    const int nparts = mode == CHAIN_FWD_OUT ? D / VW : 2 * NHALF;
    const int hv = int(blockIdx.x % unsigned(nparts)), rest = int(blockIdx.x / unsigned(nparts));
    const int h = rest % p.H, n = p.doc_order[rest / p.H];
    const bool fwd = mode == CHAIN_FWD_OUT;
    const bool fragX = !fwd && hv < 2;
    const bool want_o = fwd && p.o != nullptr;
    const int col0 = (hv % (D / VW)) * VW;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = tc::align1024(smraw);
    // A1 in, K in, MMA1 done, MMA2 / MMA3 done (+48: spare barrier of the abort path)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_BAR + 36);
    // leave-the-loop decision per barrier of a step: thread 0 copies the abort flag into slot 0 / 1
    // after its wait that precedes the barrier and every thread reads that slot after the barrier,
    // so all warps leave together (a flag raised later is seen at the next barrier)
    volatile int* stopf = reinterpret_cast<volatile int*>(sm + OFF_BAR + 40);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int qd = w & 3, cc = VPT * (w >> 2);
    const int row = 32 * qd + lane;  // accumulator row (key for S / D2, token for D1)
    constexpr int LD = 96;           // the thread that issues the TMA loads
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;
    if (*p.status == KDA_ERR_DEVICE_CHECK) return;  // a failed device-side check of this call
    // 64-column blocks store the saved S_c and Delta_c straight from their shared operand tiles
    // (one TMA store per tile, issued by thread 0) instead of one row per thread
    const bool tsave = VW == 64 && fwd && p.sS != nullptr;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) tc::mbar_init(&bar[i], 1);
        *abort_flag = 0;
        stopf[0] = stopf[1] = 0;
        tc::fence_mbar_init();
        if (c0 < c1) {
            tc::tma_prefetch_map(&tm.m128);
            tc::tma_prefetch_map(&tm.m64);
        }
    }
    constexpr bool W64 = VW == 64;  // lo planes in their own tiles (else beside hi, at column VW)
    constexpr uint32_t TCOLS = W64 ? 256 : 128;
    if (w == 0) tc::tmem_alloc(tslot, TCOLS);
    for (int i = tid; i < 8192 / 16; i += CHAIN_THREADS)
        reinterpret_cast<uint4*>(sm + OFF_PAD)[i] = make_uint4(0u, 0u, 0u, 0u);

    float Sr[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int val = col0 + cc + j;
        float v0 = 0.f;
        if (!fwd) v0 = (fragX && row == val) ? 1.f : 0.f;
        else if (p.h0) v0 = p.h0[dh + size_t(row) * D + val];
        Sr[j] = v0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tslot;
    // TMEM columns: D1 0..2 VW - 1 (two halves), D2 from 128 (64-column blocks) or 64
    const uint32_t tD1 = taddr + (uint32_t(32 * qd) << 16), tD2 = tD1 + (W64 ? 128 : 64);

    const uint32_t ID1 = tc::idesc_bf16(128, VW, false, true);  // K-major A, MN-major B
    const uint32_t ID2 = tc::idesc_bf16(128, VW, true, true);   // MN-major A and B
    const uint32_t ID1c = tc::idesc_bf16(128, 2 * VW, false, true), ID2c = tc::idesc_bf16(128, 2 * VW, true, true);
    // sum of the two column halves of an accumulator
    auto tld = [&](uint32_t tcol, float (&v)[VPT]) {
        float v2[VPT];
        tc::tmem_ld<VPT>(tcol, v);
        tc::tmem_ld<VPT>(tcol + VW, v2);
#pragma unroll
        for (int j = 0; j < VPT; ++j) v[j] += v2[j];
    };
    const uint32_t sA1 = smem_u32(sm + OFF_A1), sS = smem_u32(sm + OFF_S);
    const uint32_t sKt = smem_u32(sm + OFF_KT), sPad = smem_u32(sm + OFF_PAD);
    const uint32_t sDl = smem_u32(sm + OFF_DL);

    const uint32_t bytesA1 = want_o ? 65536u : 32768u, bytesK = want_o ? 49152u : 32768u;
    // one TMA operation per operand image (each costs the issuing thread ~100+ cycles)
    auto load_A1 = [&](int ci) {
        const int chd = ci * p.H + h;
        tc::mbar_expect_tx(&bar[0], bytesA1);
        if (want_o) {  // [W; Qg] per plane: {columns, rows, W / Qg, column block}
            tc::tma5(sm + OFF_A1, &tm.mA1, 0, 0, 0, 0, tm.zWh + chd, &bar[0]);
            tc::tma5(sm + OFF_A1 + 32768, &tm.mA1, 0, 0, 0, 0, tm.zWl + chd, &bar[0]);
        } else {  // W rows only (rows 64..127 of the operand are not read back)
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tc::tma3(sm + OFF_A1 + kb * 16384, &tm.m128, 64 * kb, 0, tm.zWh + chd, &bar[0]);
                tc::tma3(sm + OFF_A1 + 32768 + kb * 16384, &tm.m128, 64 * kb, 0, tm.zWl + chd, &bar[0]);
            }
        }
    };
    auto load_K = [&](int ci) {
        const int chd = ci * p.H + h;
        tc::mbar_expect_tx(&bar[1], bytesK);
        tc::tma5(sm + OFF_KT, &tm.mKb, 0, 0, 0, 0, tm.zKh + chd, &bar[1]);
        if (want_o) tc::tma4(sm + OFF_AQ, &tm.mAq, 0, 0, 0, tm.zAh + chd, &bar[1]);
    };
    // per-thread operands of the next chunk, fetched one chunk ahead: its U row (lanes 0..63),
    // e^gL of this thread's key, its chunk-table entry
    float Un[VPT];
    float egn = 0.f;
    int4 infon = make_int4(0, 0, 0, 0);
    auto fetch_next = [&](int ci) {
        if (ci >= c1) return;
        const size_t chd = size_t(ci) * p.H + h;
        if (qd < 2 && !fragX) {
            const float4* src = reinterpret_cast<const float4*>(p.U + chd * CH * D + size_t(row) * D + col0 + cc);
#pragma unroll
            for (int j = 0; j < VPT / 4; ++j) {
                const float4 u4 = src[j];
                Un[4 * j] = u4.x;
                Un[4 * j + 1] = u4.y;
                Un[4 * j + 2] = u4.z;
                Un[4 * j + 3] = u4.w;
            }
        }
        egn = p.eGL[chd * D + row];
        infon = p.chunk_tab[ci];
    };
#pragma unroll
    for (int j = 0; j < VPT; ++j) Un[j] = 0.f;
    fetch_next(c0);

    // phase parity of the latest loads (the loader thread's bookkeeping for an early exit: a wait
    // on it returns at once when they have landed), -1 = none
    int pendA = -1, pendK = -1;
    if (tid == LD && c0 < c1) {
        load_A1(c0);
        load_K(c0);
        pendA = pendK = 0;
    }

    for (int ci = c0; ci < c1; ++ci) {
        const uint32_t ph = uint32_t(ci - c0) & 1u;
        const size_t chd = size_t(ci) * p.H + h;
        uint32_t sh[VPT / 2], sl[VPT / 2];
        tc::split_n<VPT>(Sr, sh, sl);
        tc::st_sw128_n<VPT>(sm + OFF_S, row, cc, sh);
        tc::st_sw128_n<VPT>(sm + OFF_S + (W64 ? 16384 : 0), row, (W64 ? 0 : VW) + cc, sl);
        tc::fence_async_smem();
        // the previous chunk's Delta store has read its tile (rewritten below this barrier)
        if (tsave && tid == 0) tc::bulk_wait_read0();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (stopf[0]) break;

        // ---- MMA1: D1 = [W; Qg] S ----
        if (tid == 0) {
            if (tc::mbar_wait(&bar[0], ph)) {
                tc::fence_after_sync();
                const uint64_t dAh = tc::sdesc(sA1, 16, 1024), dAl = tc::sdesc(sA1 + 32768, 16, 1024);
                const uint64_t dSh = tc::sdesc(sS, 1024, 1024);
                const uint64_t dShl = tc::sdesc(sS, W64 ? 16384 : 1024, 1024);  // [hi | lo] along N
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint64_t ak = uint64_t(((s >> 2) * 16384 + (s & 3) * 32) >> 4);
                    const uint64_t bk = uint64_t((s * 2048) >> 4);
                    tc::mma(taddr, dAh + ak, dShl + bk, ID1c, s > 0 ? 1u : 0u);
                    tc::mma(taddr, dAl + ak, dSh + bk, ID1, 1u);
                }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[2]);
            if (tsave) {  // the saved start state, both planes, from the S tile
                tc::tma_store3(&tm.mSst, col0, 0, int(2 * chd), sm + OFF_S);
                tc::bulk_commit();
            }
        }
        __syncwarp();
        // while MMA1 runs: the saved start state, this chunk's U row and e^gL
        if (fwd && p.sS && !tsave) {
            __nv_bfloat16* dst = p.sS + chd * 2 * D * D + size_t(row) * D + col0 + cc;
            tc::st_g_n<VPT>(dst, sh);
            tc::st_g_n<VPT>(dst + D * D, sl);
        }
        const float eg = egn;
        const int4 info = infon;
        if (!tc::mbar_wait(&bar[2], ph)) *abort_flag = 1;
        if (tid == 0) stopf[1] = *abort_flag;  // decision at the next barrier
        tc::fence_after_sync();
        if (tid == LD && ci + 1 < c1 && !*abort_flag) {
            load_A1(ci + 1);
            pendA = int(ph ^ 1u);
        }
        __syncwarp();

        // ---- Delta = U - W S (lanes 0..63) ----
        uint32_t dhh[VPT / 2], dll[VPT / 2];
        if (qd < 2) {
            float v[VPT];
            tld(tD1 + cc, v);
#pragma unroll
            for (int j = 0; j < VPT; ++j) v[j] = Un[j] - v[j];
            tc::split_n<VPT>(v, dhh, dll);
            tc::st_sw128_n<VPT>(sm + OFF_DL, row, cc, dhh);
            tc::st_sw128_n<VPT>(sm + OFF_DL + (W64 ? 8192 : 0), row, (W64 ? 0 : VW) + cc, dll);
        }
        tc::fence_async_smem();
        // this chunk's state store has read the S tile (rewritten before the next barrier)
        if (tsave && tid == 0) tc::bulk_wait_read0();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (stopf[1]) break;

        // ---- MMA2: D2 = Kb^T Delta;  MMA3: D1 += [*; Aqk] Delta ----
        if (tid == 0) {
            if (tc::mbar_wait(&bar[1], ph)) {
                tc::fence_after_sync();
                const uint64_t dKh = tc::sdesc(sKt, 8192, 1024), dKl = tc::sdesc(sKt + 16384, 8192, 1024);
                const uint64_t dDh = tc::sdesc(sDl, 1024, 1024);
                const uint64_t dDhl = tc::sdesc(sDl, W64 ? 8192 : 1024, 1024);  // [hi | lo] along N
                const uint64_t dQh = tc::sdesc(sPad, 16, 1024), dQl = tc::sdesc(sPad + 8192, 16, 1024);
                const uint32_t d2 = taddr + (W64 ? 128 : 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t kk = uint64_t((s * 2048) >> 4);
                    tc::mma(d2, dKh + kk, dDhl + kk, ID2c, s > 0 ? 1u : 0u);
                    tc::mma(d2, dKl + kk, dDh + kk, ID2, 1u);
                }
                if (want_o) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t qk = uint64_t((s * 32) >> 4), kk = uint64_t((s * 2048) >> 4);
                        tc::mma(taddr, dQh + qk, dDhl + kk, ID1c, 1u);
                        tc::mma(taddr, dQl + qk, dDh + kk, ID1, 1u);
                    }
                }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[3]);
            if (tsave) {  // the saved write vectors, both planes, from the Delta tile
                tc::tma_store3(&tm.mDst, col0, 0, int(2 * chd), sm + OFF_DL);
                tc::bulk_commit();
            }
        }
        __syncwarp();
        // while MMA2 / MMA3 run: the saved write vectors and the next chunk's per-thread operands
        if (qd < 2 && fwd && p.sDelta && !tsave) {
            __nv_bfloat16* dst = p.sDelta + chd * 2 * CH * D + size_t(row) * D + col0 + cc;
            tc::st_g_n<VPT>(dst, dhh);
            tc::st_g_n<VPT>(dst + CH * D, dll);
        }
        fetch_next(ci + 1);
        if (!tc::mbar_wait(&bar[3], ph)) *abort_flag = 1;
        if (tid == 0) stopf[0] = *abort_flag;  // decision at the next step's first barrier
        tc::fence_after_sync();
        if (tid == LD && ci + 1 < c1 && !*abort_flag) {
            load_K(ci + 1);
            pendK = int(ph ^ 1u);
        }
        __syncwarp();

        // ---- S = e^gL * S + Kb^T Delta;  O rows (lanes 64..127) ----
        {
            float v[VPT];
            tld(tD2 + cc, v);
#pragma unroll
            for (int j = 0; j < VPT; ++j) Sr[j] = fmaf(eg, Sr[j], v[j]);
        }
        if (want_o && qd >= 2) {
            float v[VPT];
            tld(tD1 + cc, v);
#pragma unroll
            for (int j = 0; j < VPT; ++j) v[j] *= p.scale;
            // token rows of this lane and of its pair (lanes 2k, 2k + 1 store together)
            const int t = row - 64, te = t & ~1;
            const size_t off = (size_t(info.y + t) * p.H + h) * D + col0 + cc;
            const size_t ldt = size_t(p.H) * D;  // token stride in elements
            if (p.out_fp32) {
                tc::st_rows_paired_f32<VPT>(static_cast<float*>(p.o) + off, ldt, v, lane,
                                            te < info.z, te + 1 < info.z);
            } else {
                uint4 c[VPT / 8];
#pragma unroll
                for (int j = 0; j < VPT / 8; ++j)
                    c[j] = make_uint4(pack2(v[8 * j], v[8 * j + 1]), pack2(v[8 * j + 2], v[8 * j + 3]),
                                      pack2(v[8 * j + 4], v[8 * j + 5]), pack2(v[8 * j + 6], v[8 * j + 7]));
                if constexpr (VPT >= 16) {
                    tc::st_rows_paired<VPT / 8>(
                        reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + off), ldt / 2, c,
                        lane, te < info.z, te + 1 < info.z);
                } else if (t < info.z) {
                    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + off)[0] = c[0];
                }
            }
        }
    }

    if (tsave && tid == 0) tc::bulk_wait0();  // saved-set stores complete before the block ends
    if (*abort_flag) {
        // after a timed-out wait: let the MMAs and loads still in flight finish (bounded), report,
        // stop
        if (tid == 0) {
            tc::drain_mmas(reinterpret_cast<uint64_t*>(sm + OFF_BAR + 48), 100000000ull);
            p.status[0] = KDA_ERR_TIMEOUT;
        }
        if (tid == LD) {
            if (pendA >= 0) tc::mbar_wait(&bar[0], uint32_t(pendA), 100000000ull);
            if (pendK >= 0) tc::mbar_wait(&bar[1], uint32_t(pendK), 100000000ull);
        }
    } else {
        float* out = fwd ? p.ht : (fragX ? p.fragM : p.fragB);
        if (out) {
            float4* dst = reinterpret_cast<float4*>(out + dh + size_t(row) * D + col0 + cc);
#pragma unroll
            for (int j = 0; j < VPT / 4; ++j)
                dst[j] = make_float4(Sr[4 * j], Sr[4 * j + 1], Sr[4 * j + 2], Sr[4 * j + 3]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(taddr, TCOLS);
}


// ------------------------------------------------------------------------------------------------
// Backward state recurrence (reverse over the chunks of a document), same machinery.  Per chunk,
// with dS = dS1 (gradient at the chunk end) in registers:
//   DA = Kb dS1 (M = 128: rows 64..127 unused),  DT = Aqk^T dO (dO exact bf16: two terms)
//   dDelta = scale DT + DA                                  (lanes 0..63)
//   DQ = Qg^T dO,  DW = W^T dDelta                          (M = 128 keys)
//   dS0 = e^gL * dS1 + scale DQ - DW                        (every thread, its own key row)
// Only DA and DW lie on the serial path from one gradient to the next.  DA and DW take their B
// operand's hi and lo planes side by side along N, as in the forward.  DT and DQ do not depend
// on it: DQ is issued right behind DA (it runs while dDelta is formed), DT of the next chunk right
// behind DW (it runs while dS0 is formed), on a double-buffered Aqk / dO tile pair.
// mode CHAIN_BWD: dS from dht; writes the dS1 and dDelta planes of every chunk and dh0.
// mode CHAIN_FRAG_C: dS from zero; writes only the fragment-start gradient C (into p.fragB).
namespace {

constexpr int B_OFF_KB = 0;        // Kb K-major [plane][2 key blocks][64 tokens][128 B]     32 KB
constexpr int B_OFF_QG = 32768;    // Qg MN-major [plane][2 key blocks][64 tokens][128 B]    32 KB
constexpr int B_OFF_W = 65536;     // W MN-major, same layout                                32 KB
constexpr int B_OFF_AQ0 = 98304;   // Aqk as MN-major A of Aqk^T: [plane][64 t][128 B]       16 KB
constexpr int B_OFF_DO0 = 114688;  // dO MN-major B: [64 tokens][128 B]                        8 KB
constexpr int B_OFF_DS = 122880;   // dS1 MN-major B: [plane][128 keys][128 B]               32 KB
constexpr int B_OFF_DD = 155648;   // dDelta MN-major B: [plane][64 tokens][128 B]           16 KB
constexpr int B_OFF_AQ1 = 172032;  // second Aqk buffer                                      16 KB
constexpr int B_OFF_DO1 = 188416;  // second dO buffer                                        8 KB
constexpr int B_OFF_BAR = 196608;  // mbarriers, TMEM base address, abort flag
constexpr size_t CHAIN_BWD_TC_SMEM = B_OFF_BAR + 128 + 1024;

static_assert(CHAIN_BWD_TC_SMEM <= 232448, "tcgen05 chain shared memory above the opt-in limit");

}  // namespace


template <int VW>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    k_chain_bwd_tc(Params p, int mode, const __grid_constant__ TcMaps tm) {
    constexpr int VPT = VW / 2, NP = D / VW;  // value columns per thread, value parts
    const int hv = int(blockIdx.x % unsigned(NP)), rest = int(blockIdx.x / unsigned(NP));
    const int h = rest % p.H, n = p.doc_order[rest / p.H];
    const bool bwd = mode == CHAIN_BWD;
    const int col0 = hv * VW;
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = tc::align1024(smraw);
    // barriers: 0 Kb in, 1 / 2 Aqk + dO in (buffer 0 / 1), 3 Qg in, 4 W in, 5 DA done, 6 DW done,
    // 7 DQ done (+80: spare barrier of the abort path)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + B_OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + B_OFF_BAR + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + B_OFF_BAR + 68);
    volatile int* stopf = reinterpret_cast<volatile int*>(sm + B_OFF_BAR + 72);  // as in the forward
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int qd = w & 3, cc = VPT * (w >> 2);
    const int row = 32 * qd + lane;
    constexpr int LD = 96;  // the thread that issues the TMA loads (warp 3: no dDelta rows)
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;
    if (*p.status == KDA_ERR_DEVICE_CHECK) return;  // a failed device-side check of this call
    // 64-column blocks store dS1 and dDelta straight from their shared operand tiles (one TMA
    // store per tile, issued by thread 0) instead of one row per thread
    const bool tsave = VW == 64 && bwd;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) tc::mbar_init(&bar[i], 1);
        *abort_flag = 0;
        stopf[0] = stopf[1] = 0;
        tc::fence_mbar_init();
        if (c0 < c1) {
            tc::tma_prefetch_map(&tm.mKb);
            tc::tma_prefetch_map(&tm.mAq);
            tc::tma_prefetch_map(&tm.mdO);
        }
    }
    constexpr bool W64 = VW == 64;  // lo planes in their own tiles (else beside hi, at column VW)
    constexpr uint32_t TCOLS = W64 ? 512 : 256;
    if (w == 0) tc::tmem_alloc(tslot, TCOLS);

    float dSr[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
        dSr[j] = (bwd && p.dht) ? p.dht[dh + size_t(row) * D + col0 + cc + j] : 0.f;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tslot;
    // TMEM columns (DA and DW as two VW-column halves each): DA 0.., DT 64.., DQ 128.., DW 192..
    // (64-column blocks: DA 0..127, DW 128..255, DT 256..319, DQ 320..383)
    const uint32_t tl = taddr + (uint32_t(32 * qd) << 16);
    constexpr uint32_t cDA = 0, cDT = W64 ? 256 : 64, cDQ = W64 ? 320 : 128, cDW = W64 ? 128 : 192;
    const uint32_t tDA = tl + cDA, tDT = tl + cDT, tDQ = tl + cDQ, tDW = tl + cDW;

    const uint32_t IDA1 = tc::idesc_bf16(128, VW, false, true);  // Kb K-major, dS1 MN-major
    const uint32_t IDMN = tc::idesc_bf16(128, VW, true, true);   // MN-major A and B
    const uint32_t IDA1c = tc::idesc_bf16(128, 2 * VW, false, true), IDMNc = tc::idesc_bf16(128, 2 * VW, true, true);
    // sum of the two column halves of an accumulator
    auto tld = [&](uint32_t tcol, float (&v)[VPT]) {
        float v2[VPT];
        tc::tmem_ld<VPT>(tcol, v);
        tc::tmem_ld<VPT>(tcol + VW, v2);
#pragma unroll
        for (int j = 0; j < VPT; ++j) v[j] += v2[j];
    };
    const uint32_t sKb = smem_u32(sm + B_OFF_KB), sQg = smem_u32(sm + B_OFF_QG);
    const uint32_t sW = smem_u32(sm + B_OFF_W), sdS = smem_u32(sm + B_OFF_DS);
    const uint32_t sdD = smem_u32(sm + B_OFF_DD);
    auto aq_buf = [&](int b) { return b ? B_OFF_AQ1 : B_OFF_AQ0; };
    auto do_buf = [&](int b) { return b ? B_OFF_DO1 : B_OFF_DO0; };
    // the Aqk / dO buffer of chunk c is (c1 - 1 - c) & 1; its n-th load completes phase n & 1 of
    // that buffer's barrier
    const int tok0 = (tid == LD && c0 < c1) ? p.chunk_tab[c0].y : 0;  // first token (loader thread)

    // one TMA operation per operand image, both planes and both key blocks
    auto load_Kb = [&](int ci) {
        tc::mbar_expect_tx(&bar[0], 32768u);
        tc::tma5(sm + B_OFF_KB, &tm.mKb, 0, 0, 0, 0, tm.zKh + ci * p.H + h, &bar[0]);
    };
    auto load_AO = [&](int ci) {
        const int b = (c1 - 1 - ci) & 1;
        tc::mbar_expect_tx(&bar[1 + b], 16384u + 8192u);
        tc::tma4(sm + aq_buf(b), &tm.mAq, 0, 0, 0, tm.zAh + ci * p.H + h, &bar[1 + b]);
        tc::tma3(sm + do_buf(b), &tm.mdO, col0, h, tok0 + CH * (ci - c0), &bar[1 + b]);
    };
    auto load_Qg = [&](int ci) {
        tc::mbar_expect_tx(&bar[3], 32768u);
        tc::tma5(sm + B_OFF_QG, &tm.mKb, 0, 0, 0, 0, tm.zQh + ci * p.H + h, &bar[3]);
    };
    auto load_W = [&](int ci) {
        tc::mbar_expect_tx(&bar[4], 32768u);
        tc::tma5(sm + B_OFF_W, &tm.mKb, 0, 0, 0, 0, tm.zWh + ci * p.H + h, &bar[4]);
    };
    // DT = Aqk^T dO of chunk ci into its TMEM columns (thread 0), once its Aqk / dO buffer landed
    auto issue_DT = [&](int ci) -> bool {
        const int k = c1 - 1 - ci, b = k & 1;
        if (!tc::mbar_wait(&bar[1 + b], uint32_t(k >> 1) & 1u)) return false;
        tc::fence_after_sync();
        const uint32_t sAq = smem_u32(sm + aq_buf(b)), sdO = smem_u32(sm + do_buf(b));
        const uint64_t ah = tc::sdesc(sAq, 8192, 1024), al = tc::sdesc(sAq + 8192, 8192, 1024);
        const uint64_t bo = tc::sdesc(sdO, 1024, 1024);
        uint32_t acc = 0;
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                tc::mma(taddr + cDT, (t2 ? ah : al) + uint64_t((s * 2048) >> 4),
                        bo + uint64_t((s * 2048) >> 4), IDMN, acc);
                acc = 1;
            }
        return true;
    };
    // next chunk's e^gL of this thread's key, fetched one chunk ahead
    float egn = 0.f;
    auto fetch_next = [&](int ci) {
        if (ci >= c0) egn = p.eGL[(size_t(ci) * p.H + h) * D + row];
    };
    fetch_next(c1 - 1);
    // phase parity of the latest load per barrier 0..4 (the loader thread's bookkeeping for an
    // early exit: a wait on it returns at once when it has landed), -1 = none
    int pend[5] = {-1, -1, -1, -1, -1};
    if (tid == LD && c0 < c1) {
        load_Kb(c1 - 1);
        load_AO(c1 - 1);
        load_Qg(c1 - 1);
        load_W(c1 - 1);
        pend[0] = pend[1] = pend[3] = pend[4] = 0;
        if (c1 - 2 >= c0) {
            load_AO(c1 - 2);
            pend[2] = 0;
        }
    }
    if (tid == 0 && c0 < c1 && !issue_DT(c1 - 1)) *abort_flag = stopf[0] = 1;

    for (int ci = c1 - 1; ci >= c0; --ci) {
        const int k = c1 - 1 - ci;
        const uint32_t ph = uint32_t(k) & 1u;
        const size_t chd = size_t(ci) * p.H + h;
        uint32_t sh_[VPT / 2], sl_[VPT / 2];  // dS1 operand split (its saved planes are written below)
        tc::split_n<VPT>(dSr, sh_, sl_);
        tc::st_sw128_n<VPT>(sm + B_OFF_DS, row, cc, sh_);
        tc::st_sw128_n<VPT>(sm + B_OFF_DS + (W64 ? 16384 : 0), row, (W64 ? 0 : VW) + cc, sl_);
        tc::fence_async_smem();
        // the previous chunk's dDelta store has read its tile (rewritten below this barrier)
        if (tsave && tid == 0) tc::bulk_wait_read0();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (stopf[0]) break;

        // ---- DA = Kb dS1, then DQ = Qg^T dO ----
        if (tid == 0) {
            if (tc::mbar_wait(&bar[0], ph)) {
                tc::fence_after_sync();
                const uint64_t kh = tc::sdesc(sKb, 16, 1024), kl = tc::sdesc(sKb + 16384, 16, 1024);
                const uint64_t dh_ = tc::sdesc(sdS, 1024, 1024);
                const uint64_t dhl = tc::sdesc(sdS, W64 ? 16384 : 1024, 1024);  // [hi | lo] along N
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint64_t ak = uint64_t(((s >> 2) * 8192 + (s & 3) * 32) >> 4);
                    const uint64_t bk = uint64_t((s * 2048) >> 4);
                    tc::mma(taddr + cDA, kh + ak, dhl + bk, IDA1c, s > 0 ? 1u : 0u);
                    tc::mma(taddr + cDA, kl + ak, dh_ + bk, IDA1, 1u);
                }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[5]);
            if (tc::mbar_wait(&bar[3], ph)) {
                tc::fence_after_sync();
                const uint64_t qh = tc::sdesc(sQg, 8192, 1024), ql = tc::sdesc(sQg + 16384, 8192, 1024);
                const uint64_t bo = tc::sdesc(smem_u32(sm + do_buf(int(ph))), 1024, 1024);
                uint32_t acc = 0;
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        tc::mma(taddr + cDQ, (t2 ? qh : ql) + uint64_t((s * 2048) >> 4),
                                bo + uint64_t((s * 2048) >> 4), IDMN, acc);
                        acc = 1;
                    }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[7]);
            if (tsave) {  // the gradient at the chunk end, both planes, from the dS1 tile
                tc::tma_store3(&tm.mdSst, col0, 0, int(2 * chd), sm + B_OFF_DS);
                tc::bulk_commit();
            }
        }
        __syncwarp();
        if (bwd && !tsave) {  // while DA runs: the saved gradient at the chunk end
            __nv_bfloat16* dst = p.dS1 + chd * 2 * D * D + size_t(row) * D + col0 + cc;
            tc::st_g_n<VPT>(dst, sh_);
            tc::st_g_n<VPT>(dst + D * D, sl_);
        }
        const float eg = egn;
        if (!tc::mbar_wait(&bar[5], ph)) *abort_flag = 1;  // DA (and this chunk's DT) done
        tc::fence_after_sync();
        if (tid == LD && ci > c0 && !*abort_flag) {
            load_Kb(ci - 1);
            pend[0] = int(ph ^ 1u);
        }
        __syncwarp();

        // ---- dDelta = scale DT + DA (lanes 0..63) ----
        uint32_t xh[VPT / 2], xl[VPT / 2];
        if (qd < 2) {
            float a[VPT], t[VPT];
            tld(tDA + cc, a);
            tc::tmem_ld<VPT>(tDT + cc, t);
#pragma unroll
            for (int j = 0; j < VPT; ++j) a[j] = fmaf(p.scale, t[j], a[j]);
            tc::split_n<VPT>(a, xh, xl);
            tc::st_sw128_n<VPT>(sm + B_OFF_DD, row, cc, xh);
            tc::st_sw128_n<VPT>(sm + B_OFF_DD + (W64 ? 8192 : 0), row, (W64 ? 0 : VW) + cc, xl);
        }
        if (tid == LD) {
            if (!tc::mbar_wait(&bar[7], ph)) *abort_flag = 1;  // DQ done: the Qg buffer is free
            tc::fence_after_sync();
            if (ci > c0 && !*abort_flag) {
                load_Qg(ci - 1);
                pend[3] = int(ph ^ 1u);
            }
        }
        if (tid == 0) {
            stopf[1] = *abort_flag;  // decision at the next barrier
            if (tsave) tc::bulk_wait_read0();  // this chunk's dS1 store has read its tile
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (stopf[1]) break;

        // ---- DW = W^T dDelta, then DT of the next chunk ----
        if (tid == 0) {
            if (tc::mbar_wait(&bar[4], ph)) {
                tc::fence_after_sync();
                const uint64_t wh = tc::sdesc(sW, 8192, 1024), wl = tc::sdesc(sW + 16384, 8192, 1024);
                const uint64_t dxh = tc::sdesc(sdD, 1024, 1024);
                const uint64_t dxhl = tc::sdesc(sdD, W64 ? 8192 : 1024, 1024);  // [hi | lo] along N
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t kk = uint64_t((s * 2048) >> 4);
                    tc::mma(taddr + cDW, wh + kk, dxhl + kk, IDMNc, s > 0 ? 1u : 0u);
                    tc::mma(taddr + cDW, wl + kk, dxh + kk, IDMN, 1u);
                }
            } else {
                *abort_flag = 1;
            }
            tc::mma_commit(&bar[6]);
            if (tsave) {  // the write-vector gradient, both planes, from the dDelta tile
                tc::tma_store3(&tm.mdDst, col0, 0, int(2 * chd), sm + B_OFF_DD);
                tc::bulk_commit();
            }
            if (ci > c0 && !*abort_flag && !issue_DT(ci - 1)) *abort_flag = 1;
        }
        __syncwarp();
        // while DW runs: the saved write-vector gradient and the next chunk's per-thread operands
        if (qd < 2 && bwd && !tsave) {
            __nv_bfloat16* dst = p.dDelta + chd * 2 * CH * D + size_t(row) * D + col0 + cc;
            tc::st_g_n<VPT>(dst, xh);
            tc::st_g_n<VPT>(dst + CH * D, xl);
        }
        fetch_next(ci - 1);
        if (!tc::mbar_wait(&bar[6], ph)) *abort_flag = 1;  // DW (and DQ) done
        if (tid == 0) stopf[0] = *abort_flag;  // decision at the next step's first barrier
        tc::fence_after_sync();
        if (tid == LD && !*abort_flag) {
            if (ci > c0) {
                load_W(ci - 1);
                pend[4] = int(ph ^ 1u);
            }
            if (ci - 2 >= c0) {  // into this chunk's Aqk / dO buffer, now read by nothing
                load_AO(ci - 2);
                const int par = int(uint32_t((k + 2) >> 1) & 1u);
                if (ph) pend[2] = par;
                else pend[1] = par;
            }
        }
        __syncwarp();

        // ---- dS0 = e^gL * dS1 + scale DQ - DW ----
        {
            float q[VPT], x[VPT];
            tc::tmem_ld<VPT>(tDQ + cc, q);
            tld(tDW + cc, x);
#pragma unroll
            for (int j = 0; j < VPT; ++j) dSr[j] = fmaf(eg, dSr[j], fmaf(p.scale, q[j], -x[j]));
        }
    }

    if (tsave && tid == 0) tc::bulk_wait0();  // gradient stores complete before the block ends
    if (*abort_flag) {
        if (tid == 0) {
            tc::drain_mmas(reinterpret_cast<uint64_t*>(sm + B_OFF_BAR + 80), 100000000ull);
            p.status[0] = KDA_ERR_TIMEOUT;
        }
        if (tid == LD) {
#pragma unroll
            for (int i = 0; i < 5; ++i)
                if (pend[i] >= 0) tc::mbar_wait(&bar[i], uint32_t(pend[i]), 100000000ull);
        }
    } else {
        float* out = bwd ? p.dh0 : p.fragB;
        if (out) {
            float4* dst = reinterpret_cast<float4*>(out + dh + size_t(row) * D + col0 + cc);
#pragma unroll
            for (int j = 0; j < VPT / 4; ++j)
                dst[j] = make_float4(dSr[4 * j], dSr[4 * j + 1], dSr[4 * j + 2], dSr[4 * j + 3]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(taddr, TCOLS);
}

// Launchers (the kernels are templates on the value width): the narrowest of VW = 16, 32 whose
// blocks (128 / VW per (document, head)) all fit on the SMs at once, else VW = 64; the fragment
// modes use VW = 64.
cudaError_t chain_tc_setup() {
    const void* fs[6] = {(const void*)k_chain_fwd_tc<64>, (const void*)k_chain_fwd_tc<32>,
                         (const void*)k_chain_fwd_tc<16>, (const void*)k_chain_bwd_tc<64>,
                         (const void*)k_chain_bwd_tc<32>, (const void*)k_chain_bwd_tc<16>};
    for (int i = 0; i < 6; ++i) {
        const cudaError_t e = cudaFuncSetAttribute(
            fs[i], cudaFuncAttributeMaxDynamicSharedMemorySize, int(i < 3 ? CHAIN_TC_SMEM : CHAIN_BWD_TC_SMEM));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
static int chain_width(unsigned pairs, int sms) {
    return long(pairs) * (D / 16) <= sms ? 16 : long(pairs) * (D / 32) <= sms ? 32 : 64;
}
void launch_chain_fwd_tc(const Params& p, int mode, const TcMaps& tm, unsigned pairs, int sms,
                         cudaStream_t st) {
    const int vw = mode == CHAIN_FWD_OUT ? chain_width(pairs, sms) : 64;
    if (vw == 16)
        k_chain_fwd_tc<16><<<pairs * (D / 16), CHAIN_THREADS, CHAIN_TC_SMEM, st>>>(p, mode, tm);
    else if (vw == 32)
        k_chain_fwd_tc<32><<<pairs * (D / 32), CHAIN_THREADS, CHAIN_TC_SMEM, st>>>(p, mode, tm);
    else
        k_chain_fwd_tc<64><<<pairs * (mode == CHAIN_FWD_OUT ? NHALF : 2 * NHALF), CHAIN_THREADS,
                             CHAIN_TC_SMEM, st>>>(p, mode, tm);
}
void launch_chain_bwd_tc(const Params& p, int mode, const TcMaps& tm, unsigned pairs, int sms,
                         cudaStream_t st) {
    const int vw = chain_width(pairs, sms);
    if (vw == 16)
        k_chain_bwd_tc<16><<<pairs * (D / 16), CHAIN_THREADS, CHAIN_BWD_TC_SMEM, st>>>(p, mode, tm);
    else if (vw == 32)
        k_chain_bwd_tc<32><<<pairs * (D / 32), CHAIN_THREADS, CHAIN_BWD_TC_SMEM, st>>>(p, mode, tm);
    else
        k_chain_bwd_tc<64><<<pairs * NHALF, CHAIN_THREADS, CHAIN_BWD_TC_SMEM, st>>>(p, mode, tm);
}

}  // namespace kda
