// Intra-chunk stage of the forward: per (chunk, head) the gate cumsum, the fused L2 norm, the
// 64x64 matrices Akk (strictly lower, the KK^T part of the delta rule) and Aqk (lower incl. the
// diagonal), the UT / WY inverse Minv = (I + diag(beta) Akk)^-1, W = Minv diag(beta)(K e^gam),
// U = Minv diag(beta) V, and the operands Qg = Q e^gam, Kb = K e^(gL - gam) of the recurrence.
//
// Exponent differences (secondary chunking into four 16-row sub-chunks, after Gated Linear
// Attention): for rows r of sub-chunk i and columns s of an earlier sub-chunk j the factor
// exp(gam_r - gam_s) is split at the last row e_j of sub-chunk j into exp(gam_r - gam_ej) and
// exp(gam_ej - gam_s); with a decaying gate both are <= 1, so the product runs on tensor cores
// without overflow at any decay rate.  Inside a sub-chunk (the diagonal 16x16 blocks) the factor
// is formed elementwise in FP32.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int LB = 136;  // row stride (bf16 elements) of [rows][128] MMA operand tiles
// row stride (floats) of the q, k, gam tiles: 8 words of bank offset per row, so the 8-byte
// fragment reads of step 4c (rows g, columns 2t of a quad-lane layout) meet no bank conflict
constexpr int LQ = D + 8;
// row stride (floats) of the 64 x 64 tiles Akk, Aqk, Minv: 16-byte aligned rows (8-byte fragment
// and staging reads) and 4 banks per row (the G and X phases' column-wise B reads meet no conflict)
constexpr int LA = CH + 4;

// The base is 1024-byte aligned; so are q, k, x, u and v, which double as 128-byte-swizzled tiles
// of the tensor-memory accelerator: after step 5 Aqk / Minv hi / lo in k (TMA store sources; Minv
// also the A operand of W) and Akk in x.akk_st, Minv diag(beta) hi / lo in q (A operand of U),
// beta K e^gam hi / lo in u and V in v (B operands of W and U); after step 6 W hi / lo in u (TMA
// store source until the next item's step 4a).
struct IntraSmem {
    float q[CH * LQ], k[CH * LQ], gam[CH * LQ];
    union {
        unsigned char akk_st[2 * 8192];  // Akk staged for its TMA store: boxes [64 rows][32 fp32]
        float P[6][16 * 32];             // partial sums of step 4 (dead before step 5)
        uint4 gfrag[6 * 2 * 32];         // split A fragments of G_il (step 5): [pair][hi, lo][lane]
    } x;
    union {
        struct {
            __nv_bfloat16 Ks[3][2][16 * LB];  // B operands of the off-diagonal blocks (hi, lo)
        } a;
        // beta K e^gam (hi, lo) as the MN-major B operand of W: [plane][column block of 64][64
        // token rows][128 bytes], written during step 5
        unsigned char bkg[2 * 16384];
        unsigned char wst[4 * 8192];  // W staged: boxes [plane][column block] of 64 rows x 64 bf16
    } u;
    unsigned char v[2 * 8192];  // V (exact in bf16), MN-major B of U: [column block][64 rows][128 B]
    float Akk[CH * LA], Aqk[CH * LA], Mi[CH * LA];
    float beta[CH];
    uint64_t mbar[3];  // 0: completion of step 6's MMAs; 1: spare of the abort path; 2: gate tile loaded
    uint32_t tslot;    // TMEM base address
    int abort;         // a bounded wait timed out
};

// off-diagonal sub-chunk pairs (i, j), i > j, one per warp
__constant__ int2 kPairs[6] = {{1, 0}, {2, 0}, {3, 0}, {2, 1}, {3, 1}, {3, 2}};


static_assert(sizeof(IntraSmem) + 1024 <= 232448, "intra shared memory above the opt-in limit");
static_assert(offsetof(IntraSmem, Akk) % 16 == 0 && (CH * LA) % 4 == 0,
              "the 64 x 64 tiles are cleared with 16-byte stores");
static_assert(offsetof(IntraSmem, gam) % 128 == 0, "the gate tile is a TMA destination");
static_assert(offsetof(IntraSmem, k) % 1024 == 0 && offsetof(IntraSmem, x) % 1024 == 0 &&
                  offsetof(IntraSmem, u) % 1024 == 0 && offsetof(IntraSmem, v) % 1024 == 0 &&
                  CH * LQ * 4 >= 4 * 8192,
              "operand / staging tiles must be 1024-byte aligned and hold four boxes");
// (rows 64..127 of step 6's M = 128 A operands read the 8 KB after each 64-row tile: the next
// tile or the next member of this image, never past it; those accumulator rows are not read)

// Byte offset of (row, byte) inside a box of 64 rows x 128 bytes in the TMA unit's 128-byte
// swizzle: the 16-byte chunk j of row r sits at chunk position j ^ (r % 8).
__device__ __forceinline__ int sw128(int row, int byte) {
    return row * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ float4 row4(const float* t, int r, int c4) {
    return *reinterpret_cast<const float4*>(t + r * LQ + c4);
}
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}

// Partial sums over this lane's channels (cbase + 32 j + 0..3, j = 0, 1) of the diagonal 8 x 8
// block starting at row b0, for rows RB = 7 - RP (pairs s = RB..0, slots 0..RB) and RA = RP
// (pairs s = RA..0, slots RB+1..8): akk = sum_c k_r E k_s, aqk = sum_c q_r E k_s with
// E = exp(gam_r - gam_s) built as the running product of per-token decays (each <= 1).
template <int RP>
__device__ __forceinline__ void diag_pair_sums(const float* q, const float* k, const float* gam,
                                               int b0, int cbase, float (&akk)[9], float (&aqk)[9]) {
    constexpr int RB = 7 - RP, RA = RP;
#pragma unroll
    for (int j = 0; j < 9; ++j) akk[j] = aqk[j] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int c4 = cbase + 32 * j;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int R = pass == 0 ? RB : RA, slot0 = pass == 0 ? 0 : RB + 1;
            const float4 kr = row4(k, b0 + R, c4), qr = row4(q, b0 + R, c4);
            float4 gs = row4(gam, b0 + R, c4);
            float4 E = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
            for (int s = R; s >= 0; --s) {
                const float4 ks = row4(k, b0 + s, c4);
                const float4 x = make_float4(E.x * ks.x, E.y * ks.y, E.z * ks.z, E.w * ks.w);
                akk[slot0 + R - s] = dot4(kr, x, akk[slot0 + R - s]);
                aqk[slot0 + R - s] = dot4(qr, x, aqk[slot0 + R - s]);
                if (s > 0) {
                    const float4 gp = row4(gam, b0 + s - 1, c4);
                    E.x *= __expf(gs.x - gp.x);
                    E.y *= __expf(gs.y - gp.y);
                    E.z *= __expf(gs.z - gp.z);
                    E.w *= __expf(gs.w - gp.w);
                    gs = gp;
                }
            }
        }
    }
}

}  // namespace

size_t intra_smem_bytes() { return sizeof(IntraSmem) + 1024; }  // + alignment slack of the base

// Persistent: one block per SM walks the (chunk, head) items item = chunk * H + head.  The next
// item's q and k are loaded into registers in two bursts (so no burst fills the memory request
// queue of the SM), its gate tile by one TMA copy and its v tile by cp.async while the current
// item is computed; while the current item's step-6 MMAs run, the block prepares the next item's
// gate rows and clears its 64 x 64 tiles.  The hi / lo planes of Aqk, Minv and W and Akk leave
// through TMA stores from staging tiles (lane 0 of one warp per store issues it and waits for its
// reads of shared memory before the tile is rewritten, so the issue costs overlap): the small
// matrices' stores run during step 6, W's during the next item's first steps.  Step 6 (W and U)
// runs as tcgen05 MMAs issued by thread 0 into 256 TMEM columns held for the whole kernel; every
// wait on their completion is bounded (on expiry the block reports KDA_ERR_TIMEOUT, lets its MMAs
// drain, frees its TMEM and stops).
__global__ void __launch_bounds__(INTRA_THREADS, 1) k_intra_fwd(Params p, const __grid_constant__ TcMaps tm) {
    constexpr int BT = INTRA_THREADS, NW = BT / 32;
    extern __shared__ __align__(16) unsigned char smraw[];
    // 1024-byte aligned base (offset arithmetic on the shared array keeps its address space known)
    IntraSmem& S = *reinterpret_cast<IntraSmem*>(smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int items = *p.nchunks * p.H;
    const int c4t = (tid & 31) * 4;  // the gate channels of this thread (every k below)

    // raw inputs of the next item (rows past the document end read as zero): q, k, beta in
    // registers; the gate and v go to their shared tiles with cp.async once the current item no
    // longer needs them (gam after step 5, v after step 6)
    uint4 pq[2], pk[2];
    float4 pdb = make_float4(0.f, 0.f, 0.f, 0.f);
    float pb = 0.f, peA = 0.f;
    int nT0 = 0, nL = 0, nh = 0;  // first token, length and head of the next item
    int4 tab_ahead = make_int4(0, 0, 0, 0);  // chunk-table entry of the item after the next
    // parts: bit 0 q, bit 1 k, bit 2 gate (one TMA copy into gam, rows dense, issued by thread 0) /
    // beta / gate parameters / next chunk-table entry
    auto fetch = [&](int item, int4 inf, int parts) {
        const int hh = item % p.H;
        const int T0 = inf.y, Ln = inf.z;
        nT0 = T0;
        nL = Ln;
        nh = hh;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = tid + BT * k, r = i >> 4, c8 = (i & 15) * 8;
            const size_t off = (size_t(T0 + r) * p.H + hh) * D + c8;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            if (parts & 1) pq[k] = r < Ln ? *reinterpret_cast<const uint4*>(p.q + off) : z;
            if (parts & 2) pk[k] = r < Ln ? *reinterpret_cast<const uint4*>(p.k + off) : z;
        }
        if (!(parts & 4)) return;
        if (tid == 0) {  // rows past the document end are zeroed in step 1
            tc::fence_async_smem();  // the tile's earlier generic accesses come first
            tc::mbar_expect_tx(&S.mbar[2], CH * D * 4u);
            tc::tma3(S.gam, &tm.mg, 0, hh, T0, &S.mbar[2]);
        }
        if (tid < CH) pb = tid < Ln ? bf2f(p.beta[size_t(T0 + tid) * p.H + hh]) : 0.f;
        if (p.gate_raw) {
            pdb = *reinterpret_cast<const float4*>(p.dt_bias + hh * D + c4t);
            peA = p.A_log[hh];
        }
        const int after = item + int(gridDim.x);
        if (after < items) tab_ahead = p.chunk_tab[after / p.H];
    };
    auto fetch_v = [&]() {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = tid + BT * k, r = i >> 4, c8 = (i & 15) * 8;
            const bool ok = r < nL;
            cp16z(S.v + (c8 >> 6) * 8192 + sw128(r, (c8 & 63) * 2),
                  p.v + (size_t(nT0 + (ok ? r : 0)) * p.H + nh) * D + c8, ok);
        }
        cp_commit();
    };
    if (tid == 0) {
        tc::mbar_init(&S.mbar[0], 1);
        tc::mbar_init(&S.mbar[2], 1);
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&S.tslot, 256);  // W in columns 0..127, U in 128..255
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = S.tslot;
    uint32_t mph = 0, gph = 0;  // phase parities of the MMA and gate barriers
    // An item's gate rows in place (dense tile: g, or the raw form's -exp(A_log) softplus(a +
    // dt_bias); zero past the document end) and its cleared 64 x 64 accumulators, done before its
    // step 1 -- for every item but the first while the previous item's step-6 MMAs run.
    auto prep = [&](int Ln) {
        for (int i = tid; i < CH * LA / 4; i += BT) {  // (each tile is 16-byte aligned, 4352 floats)
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4*>(S.Akk)[i] = z;
            reinterpret_cast<float4*>(S.Aqk)[i] = z;
            reinterpret_cast<float4*>(S.Mi)[i] = z;
        }
        const float eA = p.gate_raw ? expf(peA) : 0.f;
        bool bad_gate = false;
        if (!tc::mbar_wait(&S.mbar[2], gph)) S.abort = 1;  // the gate tile (dense rows)
        gph ^= 1u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = (tid + BT * k) >> 5;
            float4* g4p = reinterpret_cast<float4*>(&S.gam[r * D + c4t]);
            const float4 g4 = *g4p;
            float x[4] = {g4.x, g4.y, g4.z, g4.w};
            const float b4[4] = {pdb.x, pdb.y, pdb.z, pdb.w};
            if (p.gate_raw) {
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = r < Ln ? -eA * softplus_f(x[j] + b4[j]) : 0.f;
            } else {
                // the exponent-difference factorisation needs a decaying gate: g <= 0 (NaN fails)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[j] = r < Ln ? x[j] : 0.f;
                    bad_gate |= !(x[j] <= 0.f);
                }
            }
            *g4p = make_float4(x[0], x[1], x[2], x[3]);  // this thread's own elements
        }
        // reported in the status word; the state recurrences and backward kernels of this call
        // then do nothing
        if (bad_gate) p.status[0] = KDA_ERR_DEVICE_CHECK;
    };
    if (int(blockIdx.x) < items) {
        fetch(blockIdx.x, p.chunk_tab[blockIdx.x / p.H], 7);
        fetch_v();
        prep(nL);
    }

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const size_t chd = size_t(item);

    // 1. inputs (fetched one item ahead) to shared memory, gate, beta
    float4 gx[4];  // this thread's gate values (rows w + 16 k), written to the padded tile after
                   // the barrier below (every dense row has been read by then)
    {
        if (tid < CH) S.beta[tid] = pb;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = tid + BT * k, r = i >> 4, c8 = (i & 15) * 8;
            const __nv_bfloat162* bq = reinterpret_cast<const __nv_bfloat162*>(&pq[k]);
            const __nv_bfloat162* bk = reinterpret_cast<const __nv_bfloat162*>(&pk[k]);
            float fq[8], fk[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 a = __bfloat1622float2(bq[j]), b = __bfloat1622float2(bk[j]);
                fq[2 * j] = a.x;
                fq[2 * j + 1] = a.y;
                fk[2 * j] = b.x;
                fk[2 * j + 1] = b.y;
            }
            float4* dq = reinterpret_cast<float4*>(&S.q[r * LQ + c8]);
            float4* dk = reinterpret_cast<float4*>(&S.k[r * LQ + c8]);
            dq[0] = make_float4(fq[0], fq[1], fq[2], fq[3]);
            dq[1] = make_float4(fq[4], fq[5], fq[6], fq[7]);
            dk[0] = make_float4(fk[0], fk[1], fk[2], fk[3]);
            dk[1] = make_float4(fk[4], fk[5], fk[6], fk[7]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) gx[k] = *reinterpret_cast<const float4*>(&S.gam[((tid + BT * k) >> 5) * D + c4t]);
    }
    __syncthreads();
    const bool more = item + int(gridDim.x) < items;
#pragma unroll
    for (int k = 0; k < 4; ++k) *reinterpret_cast<float4*>(&S.gam[((tid + BT * k) >> 5) * LQ + c4t]) = gx[k];

    // 2. fused L2 norm (warp per row)
    if (p.l2n) {
        for (int r = warp; r < CH; r += NW) {
            float a = 0.f, b = 0.f;
            for (int c = lane; c < D; c += 32) {
                const float x = S.q[r * LQ + c], y = S.k[r * LQ + c];
                a = fmaf(x, x, a);
                b = fmaf(y, y, b);
            }
            a = warp_sum(a);
            b = warp_sum(b);
            const float ra = 1.f / sqrtf(a + p.eps), rb = 1.f / sqrtf(b + p.eps);
            for (int c = lane; c < D; c += 32) {
                S.q[r * LQ + c] *= ra;
                S.k[r * LQ + c] *= rb;
            }
        }
    }
    __syncthreads();  // the gate rows in the padded tile
    // 3. in-chunk inclusive cumsum: four threads per channel (16 rows each), then carries
    {
        const int c = tid & (D - 1), qu = tid >> 7, r0 = 16 * qu;
        float run = 0.f;
#pragma unroll
        for (int r = r0; r < r0 + 16; ++r) {
            run += S.gam[r * LQ + c];
            S.gam[r * LQ + c] = run;
        }
        __syncthreads();
        float carry = 0.f;
        for (int q2 = 0; q2 < qu; ++q2) carry += S.gam[(16 * q2 + 15) * LQ + c];
        __syncthreads();
        if (qu > 0)
#pragma unroll
            for (int r = r0; r < r0 + 16; ++r) S.gam[r * LQ + c] += carry;
    }
    if (warp >= NW - 4 && lane == 0) tc::bulk_wait_read0();  // the previous item's W stores have read u (written in 4a)
    __syncthreads();

    // 4a. diagonal 8x8 blocks (the lower-left 8x8 quadrant of each 16-row sub-chunk runs on tensor
    //     cores in 4c).  Warp = (row pair rp: rows 7 - rp and rp, blocks 4 bq..4 bq + 3, channel
    //     half chh), lane = (block, 8-channel group): every lane of a warp runs the same rows, so
    //     the running products need no divergent control flow.  Channel groups are summed with
    //     shuffles, the two channel halves through shared scratch, both in a fixed order.
    {
        const int rp = warp & 3, bq = (warp >> 2) & 1, chh = warp >> 3;
        const int b = 4 * bq + (lane >> 3), cg = lane & 7;
        float akk[9], aqk[9];
        switch (rp) {
            case 0: diag_pair_sums<0>(S.q, S.k, S.gam, 8 * b, 64 * chh + 4 * cg, akk, aqk); break;
            case 1: diag_pair_sums<1>(S.q, S.k, S.gam, 8 * b, 64 * chh + 4 * cg, akk, aqk); break;
            case 2: diag_pair_sums<2>(S.q, S.k, S.gam, 8 * b, 64 * chh + 4 * cg, akk, aqk); break;
            default: diag_pair_sums<3>(S.q, S.k, S.gam, 8 * b, 64 * chh + 4 * cg, akk, aqk); break;
        }
#pragma unroll
        for (int j = 0; j < 9; ++j)
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                akk[j] += __shfl_xor_sync(0xffffffffu, akk[j], o);
                aqk[j] += __shfl_xor_sync(0xffffffffu, aqk[j], o);
            }
        float* part = &S.x.P[0][0];  // [channel half][block][row pair][9 akk | 9 aqk]
        if (cg == 0) {
#pragma unroll
            for (int j = 0; j < 9; ++j) {
                part[((chh * 8 + b) * 4 + rp) * 18 + j] = akk[j];
                part[((chh * 8 + b) * 4 + rp) * 18 + 9 + j] = aqk[j];
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < 8 * 4 * 9; idx += BT) {
        const int b = idx / 36, rp = (idx / 9) % 4, j = idx % 9;
        const int rB = 7 - rp, rA = rp;
        const bool rowB = j <= rB;
        const int r = 8 * b + (rowB ? rB : rA), sc = 8 * b + (rowB ? rB - j : rA - (j - rB - 1));
        const float* p0 = &S.x.P[0][0] + (b * 4 + rp) * 18;
        const float* p1 = p0 + 8 * 4 * 18;
        if (sc < r) S.Akk[r * LA + sc] = p0[j] + p1[j];
        S.Aqk[r * LA + sc] = p0[9 + j] + p1[9 + j];
    }
    // 4b. B operands Ks_j[sl][c] = k[16j+sl][c] exp(gam[16j+15][c] - gam[16j+sl][c]), j = 0..2
    for (int idx = tid; idx < 3 * 16 * D / 4; idx += BT) {  // four channels per pass
        const int j = idx / (4 * D), rem = idx % (4 * D), sl = rem / (D / 4), c = (rem % (D / 4)) * 4;
        const int s = 16 * j + sl, e = 16 * j + 15;
        const float4 kv = row4(S.k, s, c), ge = row4(S.gam, e, c), gs = row4(S.gam, s, c);
        uint32_t h0, l0, h1, l1;
        split2(kv.x * __expf(ge.x - gs.x), kv.y * __expf(ge.y - gs.y), h0, l0);
        split2(kv.z * __expf(ge.z - gs.z), kv.w * __expf(ge.w - gs.w), h1, l1);
        *reinterpret_cast<uint2*>(&S.u.a.Ks[j][0][sl * LB + c]) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(&S.u.a.Ks[j][1][sl * LB + c]) = make_uint2(l0, l1);
    }
    __syncthreads();
    // 4c. off-diagonal blocks on tensor cores: warp w < 12 takes pair w / 2 and half w % 2 of the
    //     128 channels (k-steps); the two halves are added in a fixed order.  Warps 12..15 take the
    //     lower-left 8x8 quadrant of sub-chunk b = w - 12 (rows 16b+8.., columns 16b..16b+7),
    //     split at the quadrant boundary e = 16b+7 so both factors are <= 1.
    if (warp >= 12) {
        const int b = warp - 12, e = 16 * b + 7;
        float accQ[4] = {}, accK[4] = {};
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t qh[4] = {}, ql[4] = {}, kh4[4] = {}, kl[4] = {};
#pragma unroll
            for (int rr = 1; rr < 4; rr += 2) {  // rows 16b + 8 + g; rows 16b + g stay zero
                const int row = 16 * b + 8 + g, col = 16 * ks + 2 * t + 8 * (rr >> 1);
                const float2 gr = *reinterpret_cast<const float2*>(&S.gam[row * LQ + col]);
                const float2 ge = *reinterpret_cast<const float2*>(&S.gam[e * LQ + col]);
                const float2 qv = *reinterpret_cast<const float2*>(&S.q[row * LQ + col]);
                const float2 kv = *reinterpret_cast<const float2*>(&S.k[row * LQ + col]);
                const float e0 = __expf(gr.x - ge.x), e1 = __expf(gr.y - ge.y);
                split2(qv.x * e0, qv.y * e1, qh[rr], ql[rr]);
                split2(kv.x * e0, kv.y * e1, kh4[rr], kl[rr]);
            }
            uint32_t bh[2], bl[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // B[k = channel][n = s]: k[s][c] exp(gam_e - gam_s)
                const int sr = 16 * b + g, c = 16 * ks + 2 * t + 8 * hf;
                const float2 gs = *reinterpret_cast<const float2*>(&S.gam[sr * LQ + c]);
                const float2 ge = *reinterpret_cast<const float2*>(&S.gam[e * LQ + c]);
                const float2 kv = *reinterpret_cast<const float2*>(&S.k[sr * LQ + c]);
                split2(kv.x * __expf(ge.x - gs.x), kv.y * __expf(ge.y - gs.y), bh[hf], bl[hf]);
            }
            mma_x3(accQ, qh, ql, bh[0], bh[1], bl[0], bl[1]);
            mma_x3(accK, kh4, kl, bh[0], bh[1], bl[0], bl[1]);
        }
#pragma unroll
        for (int e4 = 2; e4 < 4; ++e4) {
            const int row = 16 * b + 8 + g, col = 16 * b + 2 * t + (e4 & 1);
            S.Aqk[row * LA + col] = accQ[e4];
            S.Akk[row * LA + col] = accK[e4];
        }
    } else {
        const int pr = warp >> 1, kh = warp & 1;
        const int i = kPairs[pr].x, j = kPairs[pr].y, e = 16 * j + 15;
        float accQ[2][4] = {}, accK[2][4] = {};
#pragma unroll 2
        for (int ks = 4 * kh; ks < 4 * kh + 4; ++ks) {
            uint32_t qh[4], ql[4], kh4[4], kl[4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = 16 * i + g + 8 * (rr & 1), col = 16 * ks + 2 * t + 8 * (rr >> 1);
                const float2 gr = *reinterpret_cast<const float2*>(&S.gam[row * LQ + col]);
                const float2 ge = *reinterpret_cast<const float2*>(&S.gam[e * LQ + col]);
                const float2 qv = *reinterpret_cast<const float2*>(&S.q[row * LQ + col]);
                const float2 kv = *reinterpret_cast<const float2*>(&S.k[row * LQ + col]);
                const float e0 = __expf(gr.x - ge.x), e1 = __expf(gr.y - ge.y);
                split2(qv.x * e0, qv.y * e1, qh[rr], ql[rr]);
                split2(kv.x * e0, kv.y * e1, kh4[rr], kl[rr]);
            }
            uint32_t bh[4], bl[4];
            ldsm4(bh, bn_addr(S.u.a.Ks[j][0], LB, 16 * ks, 0, lane));
            ldsm4(bl, bn_addr(S.u.a.Ks[j][1], LB, 16 * ks, 0, lane));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                mma_x3(accQ[nt], qh, ql, bh[2 * nt], bh[2 * nt + 1], bl[2 * nt], bl[2 * nt + 1]);
                mma_x3(accK[nt], kh4, kl, bh[2 * nt], bh[2 * nt + 1], bl[2 * nt], bl[2 * nt + 1]);
            }
        }
        float* part = S.x.P[pr];  // upper half's partial [2 n-tiles][2 (Q, K)][4] per lane
        if (kh == 1) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    part[((nt * 2 + 0) * 4 + e4) * 32 + lane] = accQ[nt][e4];
                    part[((nt * 2 + 1) * 4 + e4) * 32 + lane] = accK[nt][e4];
                }
        }
        __syncwarp();
        named_barrier_sync(1 + pr, 64);  // the two warps of this pair
        if (kh == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int row = 16 * i + g + 8 * (e4 >> 1), col = 16 * j + 8 * nt + 2 * t + (e4 & 1);
                    S.Aqk[row * LA + col] = accQ[nt][e4] + part[((nt * 2 + 0) * 4 + e4) * 32 + lane];
                    S.Akk[row * LA + col] = accK[nt][e4] + part[((nt * 2 + 1) * 4 + e4) * 32 + lane];
                }
        }
    }
    __syncthreads();

    int4 tab_next = tab_ahead;  // (the g part below overwrites tab_ahead)
    if (more) fetch(item + gridDim.x, tab_next, 1);

    // 5. Minv = (I + diag(beta) Akk)^-1, blockwise: 16x16 diagonal inverses D_i by substitution,
    //    then on tensor cores (split-bf16 products) G_il = -D_i diag(beta_i) Akk_il for i > l and
    //    the blocks off the diagonal X_ij = sum_{l=j}^{i-1} G_il X_lj (X_jj = D_j) by increasing
    //    block distance
    if (tid >= 64) {
        // meanwhile, the other warps form step 6's operand beta K e^gam (hi, lo) (Ks, which it
        // overwrites, was consumed in step 4) and the elementwise outputs of the recurrence:
        // Qg = Q e^gam, Kb = K e^(gL - gam) (hi, lo) and gam
        __nv_bfloat16* Qh = p.Qh + chd * CH * D;
        __nv_bfloat16* Ql = p.Ql + chd * CH * D;
        __nv_bfloat16* Kh = p.Kh + chd * CH * D;
        __nv_bfloat16* Kl = p.Kl + chd * CH * D;
        float* gam = p.gam + chd * CH * D;
        if (tid - 64 < D) p.eGL[chd * D + tid - 64] = __expf(S.gam[(CH - 1) * LQ + tid - 64]);
        for (int i = tid - 64; i < CH * D / 4; i += BT - 64) {  // four channels of a row per pass
            const int r = (4 * i) / D, c = (4 * i) % D;
            const float4 kv = *reinterpret_cast<const float4*>(&S.k[r * LQ + c]);
            const float4 gv = *reinterpret_cast<const float4*>(&S.gam[r * LQ + c]);
            const float4 gl = *reinterpret_cast<const float4*>(&S.gam[(CH - 1) * LQ + c]);
            const float4 qv = *reinterpret_cast<const float4*>(&S.q[r * LQ + c]);
            const float br = S.beta[r];
            const float e0 = __expf(gv.x), e1 = __expf(gv.y), e2 = __expf(gv.z), e3 = __expf(gv.w);
            uint32_t h0, l0, h1, l1;
            split2(br * kv.x * e0, br * kv.y * e1, h0, l0);
            split2(br * kv.z * e2, br * kv.w * e3, h1, l1);
            const int bo = (c >> 6) * 8192 + sw128(r, (c & 63) * 2);
            *reinterpret_cast<uint2*>(S.u.bkg + bo) = make_uint2(h0, h1);
            *reinterpret_cast<uint2*>(S.u.bkg + 16384 + bo) = make_uint2(l0, l1);
            split2(qv.x * e0, qv.y * e1, h0, l0);
            split2(qv.z * e2, qv.w * e3, h1, l1);
            reinterpret_cast<uint2*>(Qh)[i] = make_uint2(h0, h1);
            reinterpret_cast<uint2*>(Ql)[i] = make_uint2(l0, l1);
            split2(kv.x * __expf(gl.x - gv.x), kv.y * __expf(gl.y - gv.y), h0, l0);
            split2(kv.z * __expf(gl.z - gv.z), kv.w * __expf(gl.w - gv.w), h1, l1);
            reinterpret_cast<uint2*>(Kh)[i] = make_uint2(h0, h1);
            reinterpret_cast<uint2*>(Kl)[i] = make_uint2(l0, l1);
            reinterpret_cast<float4*>(gam)[i] = gv;
        }
    } else {
        const int b = tid >> 4, cl = tid & 15, c = 16 * b + cl;
        float x[16];
#pragma unroll
        for (int rl = 0; rl < 16; ++rl) {
            const int r = 16 * b + rl;
            float acc = 0.f;
#pragma unroll
            for (int sl = 0; sl < rl; ++sl) acc = fmaf(S.Akk[r * LA + 16 * b + sl], x[sl], acc);
            x[rl] = (rl == cl) ? 1.f : -S.beta[r] * acc;
        }
#pragma unroll
        for (int rl = 0; rl < 16; ++rl) S.Mi[(16 * b + rl) * LA + c] = x[rl];
    }
    __syncthreads();
    // G_il, pair w = i (i - 1) / 2 + l on warp w < 6: A = D_i, B = diag(beta_i) Akk_il (both
    // n-tiles, so the accumulator is already G's A fragment)
    if (warp < 6) {
        const int i = warp < 1 ? 1 : warp < 3 ? 2 : 3, l = warp - i * (i - 1) / 2;
        uint32_t dh[4], dl[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = 16 * i + g + 8 * (rr & 1), col = 16 * i + 2 * t + 8 * (rr >> 1);
            const float2 m = *reinterpret_cast<const float2*>(&S.Mi[row * LA + col]);
            split2(m.x, m.y, dh[rr], dl[rr]);
        }
        float acc[2][4] = {};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t bh[2], bl[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int kr = 16 * i + 2 * t + 8 * hf, n = 16 * l + 8 * nt + g;
                split2(S.beta[kr] * S.Akk[kr * LA + n], S.beta[kr + 1] * S.Akk[(kr + 1) * LA + n],
                       bh[hf], bl[hf]);
            }
            mma_x3(acc[nt], dh, dl, bh[0], bh[1], bl[0], bl[1]);
        }
        uint32_t h[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) split2(-acc[q >> 1][2 * (q & 1)], -acc[q >> 1][2 * (q & 1) + 1], h[q], lo[q]);
        S.x.gfrag[(2 * warp) * 32 + lane] = make_uint4(h[0], h[1], h[2], h[3]);
        S.x.gfrag[(2 * warp + 1) * 32 + lane] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    __syncthreads();
    // X_ij for j = 0 .. 3 - dist, i = j + dist: warp = (j, 8-column n-tile)
#pragma unroll
    for (int dist = 1; dist < 4; ++dist) {
        if (warp < 2 * (4 - dist)) {
            const int j = warp >> 1, i = j + dist, n = 16 * j + 8 * (warp & 1) + g;
            float acc[4] = {};
#pragma unroll
            for (int l = j; l < i; ++l) {
                const int pr = i * (i - 1) / 2 + l;
                const uint4 fh = S.x.gfrag[(2 * pr) * 32 + lane], fl = S.x.gfrag[(2 * pr + 1) * 32 + lane];
                const uint32_t ah[4] = {fh.x, fh.y, fh.z, fh.w}, al[4] = {fl.x, fl.y, fl.z, fl.w};
                uint32_t bh[2], bl[2];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int kr = 16 * l + 2 * t + 8 * hf;
                    split2(S.Mi[kr * LA + n], S.Mi[(kr + 1) * LA + n], bh[hf], bl[hf]);
                }
                mma_x3(acc, ah, al, bh[0], bh[1], bl[0], bl[1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                S.Mi[(16 * i + g + 8 * (e >> 1)) * LA + 16 * j + 8 * (warp & 1) + 2 * t + (e & 1)] = acc[e];
        }
        __syncthreads();
    }

    if (more) fetch(item + gridDim.x, tab_next, 4);  // gam is free: the next item's gate

    // 7 (ahead of step 6). The small matrices, staged for TMA stores whose reads of shared memory
    //    overlap step 6: Aqk and Minv hi / lo in the k tile (boxes Ah, Al, Mh, Ml of 64 rows x 64
    //    bf16; k is not read after step 5), Akk in akk_st (the elementwise outputs were written
    //    during step 5).  Minv's planes double as the K-major A operand of W; Minv diag(beta)
    //    hi / lo, the A operand of U, go to the q tile (not read after step 5).
    {
        unsigned char* ast = reinterpret_cast<unsigned char*>(S.k);
        unsigned char* mbt = reinterpret_cast<unsigned char*>(S.q);
        for (int i = tid; i < CH * CH / 2; i += BT) {
            const int r = (2 * i) / CH, s = (2 * i) % CH, o = sw128(r, 2 * s);
            uint32_t hi, lo;
            const float2 aq = *reinterpret_cast<const float2*>(&S.Aqk[r * LA + s]);
            const float2 mi = *reinterpret_cast<const float2*>(&S.Mi[r * LA + s]);
            const float2 ak = *reinterpret_cast<const float2*>(&S.Akk[r * LA + s]);
            const float2 bs = *reinterpret_cast<const float2*>(&S.beta[s]);
            split2(aq.x, aq.y, hi, lo);
            *reinterpret_cast<uint32_t*>(ast + o) = hi;
            *reinterpret_cast<uint32_t*>(ast + 8192 + o) = lo;
            split2(mi.x, mi.y, hi, lo);
            *reinterpret_cast<uint32_t*>(ast + 2 * 8192 + o) = hi;
            *reinterpret_cast<uint32_t*>(ast + 3 * 8192 + o) = lo;
            split2(mi.x * bs.x, mi.y * bs.y, hi, lo);
            *reinterpret_cast<uint32_t*>(mbt + o) = hi;
            *reinterpret_cast<uint32_t*>(mbt + 8192 + o) = lo;
            *reinterpret_cast<float2*>(S.x.akk_st + (s >> 5) * 8192 + sw128(r, (s & 31) * 4)) = ak;
        }
    }
    cp_wait<0>();  // this item's v tile (copied during the previous item's last phase)
    if (more) fetch(item + gridDim.x, tab_next, 2);
    tc::fence_async_smem();  // this thread's staged values and operands, before the async proxy reads
    tc::fence_before_sync();
    __syncthreads();  // every thread's part of the v tile, the operands, the staged matrices
    tc::fence_after_sync();
    if (warp >= 1 && warp <= 6 && lane == 0) {  // one small-matrix store per warp, beside the MMAs
        const int b = warp - 1;
        if (b < 4) {
            const int z = b == 0 ? tm.zAh : b == 1 ? tm.zAl : b == 2 ? tm.zMh : tm.zMl;
            tc::tma_store3(&tm.m64, 0, 0, z + int(chd), reinterpret_cast<unsigned char*>(S.k) + b * 8192);
        } else {
            tc::tma_store3(&tm.mAkk, 32 * (b - 4), 0, int(chd), S.x.akk_st + (b - 4) * 8192);
        }
        tc::bulk_commit();
    }
    if (tid == 0) {
        // 6. W = Minv (beta K e^gam) (TMEM columns 0..127) and U = (Minv diag(beta)) V (columns
        //    128..255): M = 128 (rows 0..63 are the chunk's tokens, rows 64..127 are not read), N =
        //    128 channels, K = 64 tokens in four steps; A K-major (64 tokens = one 128-byte swizzle
        //    atom per row), B MN-major (two 64-channel atoms, LBO 8 KB).  W takes the split terms
        //    Minv_hi Kg_lo + Minv_lo Kg_hi + Minv_hi Kg_hi, U the terms of the two Minv diag(beta)
        //    planes against V (exact in bf16).
        const uint32_t sK = smem_u32(S.k), sQ = smem_u32(S.q), sB = smem_u32(S.u.bkg), sV = smem_u32(S.v);
        const uint64_t aMh = tc::sdesc(sK + 2 * 8192, 16, 1024), aMl = tc::sdesc(sK + 3 * 8192, 16, 1024);
        const uint64_t aBh = tc::sdesc(sQ, 16, 1024), aBl = tc::sdesc(sQ + 8192, 16, 1024);
        const uint64_t bKh = tc::sdesc(sB, 8192, 1024), bKl = tc::sdesc(sB + 16384, 8192, 1024);
        const uint64_t bV = tc::sdesc(sV, 8192, 1024);
        const uint32_t id = tc::idesc_bf16(128, 128, false, true);
        const uint64_t wa[3] = {aMh, aMl, aMh}, wb[3] = {bKl, bKh, bKh};
        uint32_t acc = 0;
#pragma unroll
        for (int t3 = 0; t3 < 3; ++t3)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                tc::mma(taddr, wa[t3] + uint64_t((ks * 32) >> 4), wb[t3] + uint64_t((ks * 2048) >> 4), id, acc);
                acc = 1;
            }
        acc = 0;
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                tc::mma(taddr + 128, (t2 ? aBh : aBl) + uint64_t((ks * 32) >> 4),
                        bV + uint64_t((ks * 2048) >> 4), id, acc);
                acc = 1;
            }
        tc::mma_commit(&S.mbar[0]);
    }
    // while the MMAs run: the next item's gate rows (landed during steps 6-7) and clears; the
    // small 64 x 64 tiles were last read by the staging pass above
    if (more) prep(nL);
    // epilogue: warps w % 4 < 2 hold the token rows (TMEM lanes 0..63), 32 columns each (w / 4):
    // U straight to global memory, W split into its staging tile (u: the MMAs have read beta K
    // e^gam by then)
    if (!tc::mbar_wait(&S.mbar[0], mph)) S.abort = 1;
    mph ^= 1u;
    tc::fence_after_sync();
    {
        const int qd = warp & 3, cq = warp >> 2;
        if (qd < 2) {
            const int r = 32 * qd + lane;
            const uint32_t tl = taddr + (uint32_t(32 * qd) << 16);
            float v[32];
            tc::tmem_ld32(tl + 128 + 32 * cq, v);
            tc::st_rows_paired_f32<32>(p.U + chd * CH * D + size_t(r) * D + 32 * cq, D, v, lane, true, true);
            tc::tmem_ld32(tl + 32 * cq, v);
            tc::st_sw128_split32(S.u.wst + (cq >> 1) * 8192, S.u.wst + 16384 + (cq >> 1) * 8192, r,
                                 32 * (cq & 1), v);
        }
    }
    tc::fence_before_sync();
    tc::fence_async_smem();
    if (warp >= 1 && warp <= 6 && lane == 0) tc::bulk_wait_read0();  // the small matrices' stores have read k, akk_st
    __syncthreads();  // W staged; every thread is done with this item's shared tiles and TMEM
    if (*reinterpret_cast<volatile int*>(&S.abort)) break;
    if (warp >= NW - 4 && lane == 0) {  // W: one store per warp
        const int b = warp - (NW - 4);
        tc::tma_store3(&tm.m128, 64 * (b & 1), 0, ((b >> 1) ? tm.zWl : tm.zWh) + int(chd), S.u.wst + b * 8192);
        tc::bulk_commit();
    }
    if (more) fetch_v();
    }
    if (tid == 0 && S.abort) {
        // after a timed-out wait (the device is already in a bad state): let this block's MMAs
        // and its gate copy in flight finish (bounded) before its TMEM is freed, report
        tc::drain_mmas(&S.mbar[1], 100000000ull);
        tc::mbar_wait(&S.mbar[2], gph, 100000000ull);
        p.status[0] = KDA_ERR_TIMEOUT;
    }
    cp_wait<0>();                    // no cp.async into the tiles is in flight past this point
    if (lane == 0) tc::bulk_wait0();  // every warp's stores are complete before the block ends
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(taddr, 256);
}

}  // namespace kda
