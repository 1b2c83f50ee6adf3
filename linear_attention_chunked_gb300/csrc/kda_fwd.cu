// Forward-side kernels: chunk plan, intra-chunk products, inter-chunk state recurrence + output.
#include "kda_internal.cuh"

namespace kda {

// Builds the chunk table from cu_seqlens on the device (no host synchronisation).  Malformed
// offsets (cu[0] != 0, decreasing, cu[N] != T) set the status word and leave zero chunks, so every
// later kernel of the call does nothing.
__global__ void k_plan(Params p) {
    __shared__ int bad;
    if (threadIdx.x == 0) {
        int b = (p.cu[0] != 0) || (int64_t(p.cu[p.N]) != p.T);
        int acc = 0;
        for (int n = 0; n < p.N; ++n) {
            int a = p.cu[n], e = p.cu[n + 1];
            if (e < a) b = 1;
            p.doc_off[n] = acc;
            int len = e > a ? e - a : 0;
            acc += (len + CH - 1) / CH;
            if (acc > p.maxC) { b = 1; acc = int(p.maxC); }
        }
        p.doc_off[p.N] = acc;
        bad = b;
        *p.nchunks = b ? 0 : acc;
        p.status[0] = b ? KDA_ERR_DEVICE_CHECK : KDA_OK;  // status of the latest call
    }
    __syncthreads();
    if (bad) {
        for (int n = threadIdx.x; n <= p.N; n += blockDim.x) p.doc_off[n] = 0;
        return;
    }
    for (int n = 0; n < p.N; ++n) {
        const int a = p.cu[n], len = p.cu[n + 1] - a, off = p.doc_off[n];
        const int nc = (len + CH - 1) / CH;
        for (int j = threadIdx.x; j < nc; j += blockDim.x)
            p.chunk_tab[off + j] = make_int4(n, a + CH * j, min(CH, len - CH * j), j);
    }
}

namespace {

constexpr int LB = 136;   // row stride (bf16) of [64][128] operand tiles
constexpr int LB64 = 72;  // row stride (bf16) of [rows][64] tiles
constexpr int LU = 68;    // row stride (fp32) of the U half tile

struct ChainFwdSmem {
    __nv_bfloat16 S[2][D * LB64];   // state S [key][64 values] (hi, lo)
    __nv_bfloat16 Dl[2][CH * LB64]; // Delta [token][64 values] (hi, lo)
    __nv_bfloat16 W[2][CH * LB];    // W [token][key]
    __nv_bfloat16 Q[2][CH * LB];    // Qg [token][key]
    __nv_bfloat16 K[2][CH * LB];    // Kb [token][key]
    __nv_bfloat16 A[2][CH * LB64];  // Aqk [token][token]
    float U[CH * LU];               // U [token][64 values]
    float eGL[D];                   // e^gL per key
};

static_assert(sizeof(ChainFwdSmem) <= 232448, "chain shared memory above the opt-in limit");

}  // namespace

size_t chain_fwd_smem_bytes() { return sizeof(ChainFwdSmem); }

// Inter-chunk state recurrence of one (document, head, 64-column value half) on tensor cores.
// Eight warps: warp w = (wq, wn) with wq = w % 4 (row group) and wn = w / 4 (32-column quarter of
// the half).  Warp w keeps keys 32 wq..32 wq+31 x columns 32 wn.. of the FP32 state in registers;
// per chunk:
//   A: Delta = U - W S            (tokens 16 wq..16 wq+15)
//   C: O = Qg S + Aqk Delta       (output; forward mode only)
//   D: S = e^gL * S + Kb^T Delta  (keys 32 wq..)
// Operands of chunk c+1 are prefetched with cp.async as soon as their buffer is consumed.
// mode CHAIN_FWD_OUT: S from h0; writes o, ht and (when p.sS) the saved S_c and Delta_c.
// mode CHAIN_FRAG_MB: blockIdx.z in 0..3: halves 0,1 evolve X = I with zero values (-> M),
//                     halves 2,3 evolve Y = 0 with the chunk values (-> B).
__global__ void __launch_bounds__(CHAIN_THREADS) k_chain_fwd(Params p, int mode) {
    constexpr int BT = CHAIN_THREADS;
    const int n = blockIdx.x, h = blockIdx.y, hv = blockIdx.z;
    const bool fwd = mode == CHAIN_FWD_OUT;
    const bool fragX = !fwd && hv < 2;
    const int col0 = (hv & 1) * 64;
    extern __shared__ __align__(16) unsigned char smraw[];
    ChainFwdSmem& sm = *reinterpret_cast<ChainFwdSmem*>(smraw);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int wq = w & 3, wn = w >> 2, cq = 32 * wn;  // row group, column quarter (local)
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;

    float Sv[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = 32 * wq + 16 * mt + g + 8 * (e >> 1);
                const int val = col0 + cq + 8 * nt + 2 * t + (e & 1);
                float v0 = 0.f;
                if (!fwd) v0 = (fragX && key == val) ? 1.f : 0.f;
                else if (p.h0) v0 = p.h0[dh + size_t(key) * D + val];
                Sv[mt][nt][e] = v0;
            }
    // writes the state's hi / lo split to shared memory (B operand of the next chunk)
    auto store_S = [&]() {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int key = 32 * wq + 16 * mt + g + 8 * hf, col = cq + 8 * nt + 2 * t;
                    uint32_t hi, lo;
                    split2(Sv[mt][nt][2 * hf], Sv[mt][nt][2 * hf + 1], hi, lo);
                    *reinterpret_cast<uint32_t*>(&sm.S[0][key * LB64 + col]) = hi;
                    *reinterpret_cast<uint32_t*>(&sm.S[1][key * LB64 + col]) = lo;
                }
    };
    auto issue_WU = [&](int ci) {
        if (ci < c1) {
            const size_t chd = size_t(ci) * p.H + h;
            cp_tile_bf16(sm.W[0], LB, p.Wh + chd * CH * D, D, CH, D, tid, BT);
            cp_tile_bf16(sm.W[1], LB, p.Wl + chd * CH * D, D, CH, D, tid, BT);
            if (!fragX) cp_tile_f32(sm.U, LU, p.U + chd * CH * D + col0, D, CH, 64, tid, BT);
        }
        cp_commit();
    };
    auto issue_QA = [&](int ci) {
        if (ci < c1 && fwd && p.o) {
            const size_t chd = size_t(ci) * p.H + h;
            cp_tile_bf16(sm.Q[0], LB, p.Qh + chd * CH * D, D, CH, D, tid, BT);
            cp_tile_bf16(sm.Q[1], LB, p.Ql + chd * CH * D, D, CH, D, tid, BT);
            cp_tile_bf16(sm.A[0], LB64, p.Ah + chd * CH * CH, CH, CH, CH, tid, BT);
            cp_tile_bf16(sm.A[1], LB64, p.Al + chd * CH * CH, CH, CH, CH, tid, BT);
        }
        cp_commit();
    };
    auto issue_K = [&](int ci) {
        if (ci < c1) {
            const size_t chd = size_t(ci) * p.H + h;
            cp_tile_bf16(sm.K[0], LB, p.Kh + chd * CH * D, D, CH, D, tid, BT);
            cp_tile_bf16(sm.K[1], LB, p.Kl + chd * CH * D, D, CH, D, tid, BT);
            cp_tile_f32(sm.eGL, D, p.eGL + chd * D, D, 1, D, tid, BT);
        }
        cp_commit();
    };
    issue_WU(c0);
    issue_QA(c0);
    issue_K(c0);
    store_S();

    for (int ci = c0; ci < c1; ++ci) {
        const int4 info = p.chunk_tab[ci];
        const int t0 = info.y, L = info.z;
        const size_t chd = size_t(ci) * p.H + h;
        // ---- A: Delta = U - W S ----
        cp_wait<2>();
        __syncthreads();
        if (fwd && p.sS) {  // saved start state of this chunk: the split in shared memory
            __nv_bfloat16* dst = p.sS + chd * 2 * D * D + col0;
            st_tile_bf16(dst, D, sm.S[0], LB64, D, 64, tid, BT);
            st_tile_bf16(dst + D * D, D, sm.S[1], LB64, D, 64, tid, BT);
        }
        float dl[4][4] = {};
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t ah[4], al[4];
            ldsm4(ah, a_addr(sm.W[0], LB, 16 * wq, 16 * ks, lane));
            ldsm4(al, a_addr(sm.W[1], LB, 16 * wq, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4t(bh, bk_addr(sm.S[0], LB64, 16 * ks, cq + 16 * np, lane));
                ldsm4t(bl, bk_addr(sm.S[1], LB64, 16 * ks, cq + 16 * np, lane));
                mma_x3(dl[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                mma_x3(dl[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = 16 * wq + g + 8 * hf, col = cq + 8 * nt + 2 * t;
                float d0 = -dl[nt][2 * hf], d1 = -dl[nt][2 * hf + 1];
                if (!fragX) {
                    d0 += sm.U[row * LU + col];
                    d1 += sm.U[row * LU + col + 1];
                }
                uint32_t hi, lo;
                split2(d0, d1, hi, lo);
                *reinterpret_cast<uint32_t*>(&sm.Dl[0][row * LB64 + col]) = hi;
                *reinterpret_cast<uint32_t*>(&sm.Dl[1][row * LB64 + col]) = lo;

            }
        __syncthreads();
        issue_WU(ci + 1);
        if (fwd && p.sDelta) {  // saved write vectors of this chunk
            __nv_bfloat16* dst = p.sDelta + chd * 2 * CH * D + col0;
            st_tile_bf16(dst, D, sm.Dl[0], LB64, CH, 64, tid, BT);
            st_tile_bf16(dst + CH * D, D, sm.Dl[1], LB64, CH, 64, tid, BT);
        }
        // ---- C: O = Qg S + Aqk Delta ----
        cp_wait<2>();
        __syncthreads();
        if (fwd && p.o) {
            float acc[4][4] = {};
#pragma unroll 2
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t ah[4], al[4];
                ldsm4(ah, a_addr(sm.Q[0], LB, 16 * wq, 16 * ks, lane));
                ldsm4(al, a_addr(sm.Q[1], LB, 16 * wq, 16 * ks, lane));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bh[4], bl[4];
                    ldsm4t(bh, bk_addr(sm.S[0], LB64, 16 * ks, cq + 16 * np, lane));
                    ldsm4t(bl, bk_addr(sm.S[1], LB64, 16 * ks, cq + 16 * np, lane));
                    mma_x3(acc[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                    mma_x3(acc[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
                }
            }
            for (int ks = 0; ks <= wq; ++ks) {  // Aqk is lower triangular
                uint32_t ah[4], al[4];
                ldsm4(ah, a_addr(sm.A[0], LB64, 16 * wq, 16 * ks, lane));
                ldsm4(al, a_addr(sm.A[1], LB64, 16 * wq, 16 * ks, lane));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bh[4], bl[4];
                    ldsm4t(bh, bk_addr(sm.Dl[0], LB64, 16 * ks, cq + 16 * np, lane));
                    ldsm4t(bl, bk_addr(sm.Dl[1], LB64, 16 * ks, cq + 16 * np, lane));
                    mma_x3(acc[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                    mma_x3(acc[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int row = 16 * wq + g + 8 * hf, col = col0 + cq + 8 * nt + 2 * t;
                    if (row < L) {
                        const size_t off = (size_t(t0 + row) * p.H + h) * D + col;
                        const float o0 = p.scale * acc[nt][2 * hf], o1 = p.scale * acc[nt][2 * hf + 1];
                        if (p.out_fp32) {
                            *reinterpret_cast<float2*>(static_cast<float*>(p.o) + off) = make_float2(o0, o1);
                        } else {
                            *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + off) = pack2(o0, o1);
                        }
                    }
                }
        }
        __syncthreads();
        issue_QA(ci + 1);
        // ---- D: S = e^gL * S + Kb^T Delta ----
        cp_wait<2>();
        __syncthreads();
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float eg = sm.eGL[32 * wq + 16 * mt + g + 8 * (e >> 1)];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) Sv[mt][nt][e] *= eg;
            }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t ah[2][4], al[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                ldsm4t(ah[mt], at_addr(sm.K[0], LB, 32 * wq + 16 * mt, 16 * ks, lane));
                ldsm4t(al[mt], at_addr(sm.K[1], LB, 32 * wq + 16 * mt, 16 * ks, lane));
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4t(bh, bk_addr(sm.Dl[0], LB64, 16 * ks, cq + 16 * np, lane));
                ldsm4t(bl, bk_addr(sm.Dl[1], LB64, 16 * ks, cq + 16 * np, lane));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma_x3(Sv[mt][2 * np], ah[mt], al[mt], bh[0], bh[1], bl[0], bl[1]);
                    mma_x3(Sv[mt][2 * np + 1], ah[mt], al[mt], bh[2], bh[3], bl[2], bl[3]);
                }
            }
        }
        __syncthreads();
        issue_K(ci + 1);
        store_S();
    }
    cp_wait<0>();
    float* out = fwd ? p.ht : (fragX ? p.fragM : p.fragB);
    if (out) {
        out += dh;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int key = 32 * wq + 16 * mt + g + 8 * hf;
                    const int val = col0 + cq + 8 * nt + 2 * t;
                    *reinterpret_cast<float2*>(out + size_t(key) * D + val) =
                        make_float2(Sv[mt][nt][2 * hf], Sv[mt][nt][2 * hf + 1]);
                }
    }
}

}  // namespace kda
