// Backward-side kernels: reverse state recurrence, per-chunk gradient products, intra-chunk
// gradients, deterministic parameter reduction.
//
// Per chunk (adjoint of the forward lines in kda_internal.cuh), with dS1 the gradient at the
// chunk-end state and dO already multiplied by the output scale:
//   dDelta = Aqk^T dO + Kb dS1                  dS0 = e^gL * dS1 + Qg^T dO - W^T dDelta
//   dR = Minv^T dDelta    dV = beta dR          P = dR S0^T      dKg = -beta P
//   dQg = dO S0^T         dKb = Delta dS1^T     dAqk = tril(dO Delta^T)
//   dM = -strict_tril(dR Delta^T)  (M = I + diag(beta) Akk)      dAkk = beta * dM
//   dbeta_r = dR_r.v_r - Kg_r.P_r + sum_{s<r} Akk[r,s] dM[r,s]
// and through the exponent differences of Aqk / Akk into q, k and gam.  The r == s terms of Aqk
// carry no gate dependence; they are left out of dgam symbolically so that they cancel exactly.
#include "kda_internal.cuh"

namespace kda {


namespace {

constexpr int LB = 136;   // row stride (bf16) of [rows][128] tiles
constexpr int LB64 = 72;  // row stride (bf16) of [rows][64] tiles

struct ChainBwdSmem {
    __nv_bfloat16 dS[2][D * LB64];   // dS [key][64 values] (hi, lo)
    __nv_bfloat16 X[2][CH * LB64];   // -dDelta [token][64 values] (hi, lo)
    __nv_bfloat16 A[2][CH * LB64];   // Aqk [token][token]
    __nv_bfloat16 K[2][CH * LB];     // Kb [token][key]
    __nv_bfloat16 Q[2][CH * LB];     // Qg [token][key]
    __nv_bfloat16 W[2][CH * LB];     // W [token][key]
    __nv_bfloat16 dO[2][CH * LB64];  // dO [token][64 values], double buffered (exact bf16)
    float eGL[D];
};

struct BwdGemmSmem {
    __nv_bfloat16 M[2][CH * LB64];   // Minv (hi, lo)
    __nv_bfloat16 X[2][CH * LB];     // dDelta (hi, lo)
    __nv_bfloat16 R[2][CH * LB];     // dR (hi, lo)
    __nv_bfloat16 S[2][D * LB];      // S_c, later dS1 [key][value] (hi, lo)
    __nv_bfloat16 O[CH * LB];        // dO (exact bf16)
    __nv_bfloat16 Dl[2][CH * LB];    // Delta (hi, lo)
};

// fp32 [rows][128] global tile -> bf16 hi/lo shared tiles with row stride LB
__device__ __forceinline__ void split_tile(__nv_bfloat16* hi, __nv_bfloat16* lo, const float* g,
                                           int rows, int tid, int nthr) {
    for (int i = tid; i < rows * D / 4; i += nthr) {
        const int r = (4 * i) / D, c = (4 * i) % D;
        const float4 v = reinterpret_cast<const float4*>(g)[i];
        uint32_t h0, l0, h1, l1;
        split2(v.x, v.y, h0, l0);
        split2(v.z, v.w, h1, l1);
        *reinterpret_cast<uint2*>(hi + r * LB + c) = make_uint2(h0, h1);
        *reinterpret_cast<uint2*>(lo + r * LB + c) = make_uint2(l0, l1);
    }
}

}  // namespace

size_t chain_bwd_smem_bytes() { return sizeof(ChainBwdSmem); }
size_t bwd_gemm_smem_bytes() { return sizeof(BwdGemmSmem); }

// Reverse state recurrence of one (document, head, 64-column value half) on tensor cores.
// Warp w keeps keys 32w..32w+31 of the FP32 gradient dS in registers; per chunk, going back:
//   A': dDelta = scale Aqk^T dO + Kb dS1     (warp w: tokens 16w..16w+15)
//   D': dS0 = e^gL * dS1 + scale Qg^T dO - W^T dDelta
// mode CHAIN_BWD: dS from dht; per chunk writes dS1 and dDelta for the per-chunk kernels; dh0.
// mode CHAIN_FRAG_C: dS from zero; writes C (= dS at the fragment start) to fragB.
__global__ void __launch_bounds__(128) k_chain_bwd(Params p, int mode) {
    const int n = blockIdx.x, h = blockIdx.y, hv = blockIdx.z;
    const bool bwd = mode == CHAIN_BWD;
    const int col0 = hv * 64;
    extern __shared__ __align__(16) unsigned char smraw[];
    ChainBwdSmem& sm = *reinterpret_cast<ChainBwdSmem*>(smraw);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;

    float dS[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = 32 * w + 16 * mt + g + 8 * (e >> 1);
                const int val = col0 + 8 * nt + 2 * t + (e & 1);
                dS[mt][nt][e] = (bwd && p.dht) ? p.dht[dh + size_t(key) * D + val] : 0.f;
            }
    auto store_dS = [&]() {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int key = 32 * w + 16 * mt + g + 8 * hf, col = 8 * nt + 2 * t;
                    uint32_t hi, lo;
                    split2(dS[mt][nt][2 * hf], dS[mt][nt][2 * hf + 1], hi, lo);
                    *reinterpret_cast<uint32_t*>(&sm.dS[0][key * LB64 + col]) = hi;
                    *reinterpret_cast<uint32_t*>(&sm.dS[1][key * LB64 + col]) = lo;
                }
    };
    // group X(ci): Aqk, Kb, dO(ci) -> dO buffer (c1-1-ci)&1 ; group Y(ci): Qg, W, e^gL
    auto issue_X = [&](int ci) {
        if (ci >= c0) {
            const int4 info = p.chunk_tab[ci];
            const size_t chd = size_t(ci) * p.H + h;
            cp_tile_bf16(sm.A[0], LB64, p.Ah + chd * CH * CH, CH, CH, CH, tid, 128);
            cp_tile_bf16(sm.A[1], LB64, p.Al + chd * CH * CH, CH, CH, CH, tid, 128);
            cp_tile_bf16(sm.K[0], LB, p.Kh + chd * CH * D, D, CH, D, tid, 128);
            cp_tile_bf16(sm.K[1], LB, p.Kl + chd * CH * D, D, CH, D, tid, 128);
            __nv_bfloat16* dst = sm.dO[(c1 - 1 - ci) & 1];
            for (int i = tid; i < CH * 8; i += 128) {
                const int r = i >> 3, c = (i & 7) * 8;
                const bool ok = r < info.z;
                const size_t row = size_t(info.y + (ok ? r : 0));
                cp16z(dst + r * LB64 + c, p.dO + (row * p.H + h) * D + col0 + c, ok);
            }
        }
        cp_commit();
    };
    auto issue_Y = [&](int ci) {
        if (ci >= c0) {
            const size_t chd = size_t(ci) * p.H + h;
            cp_tile_bf16(sm.Q[0], LB, p.Qh + chd * CH * D, D, CH, D, tid, 128);
            cp_tile_bf16(sm.Q[1], LB, p.Ql + chd * CH * D, D, CH, D, tid, 128);
            cp_tile_bf16(sm.W[0], LB, p.Wh + chd * CH * D, D, CH, D, tid, 128);
            cp_tile_bf16(sm.W[1], LB, p.Wl + chd * CH * D, D, CH, D, tid, 128);
            cp_tile_f32(sm.eGL, D, p.eGL + chd * D, D, 1, D, tid, 128);
        }
        cp_commit();
    };
    issue_X(c1 - 1);
    issue_Y(c1 - 1);
    store_dS();

    for (int ci = c1 - 1; ci >= c0; --ci) {
        const size_t chd = size_t(ci) * p.H + h;
        const __nv_bfloat16* sdO = sm.dO[(c1 - 1 - ci) & 1];
        if (bwd) {  // gradient at the chunk end
            float* dst = p.dS1 + chd * D * D;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int key = 32 * w + 16 * mt + g + 8 * hf, val = col0 + 8 * nt + 2 * t;
                        *reinterpret_cast<float2*>(dst + size_t(key) * D + val) =
                            make_float2(dS[mt][nt][2 * hf], dS[mt][nt][2 * hf + 1]);
                    }
        }
        // ---- A': dDelta = scale Aqk^T dO + Kb dS1 ----
        cp_wait<1>();
        __syncthreads();
        {
            float a1[8][4] = {}, a2[8][4] = {};
            for (int ks = w; ks < 4; ++ks) {  // Aqk^T is upper triangular
                uint32_t ah[4], al[4];
                ldsm4t(ah, at_addr(sm.A[0], LB64, 16 * w, 16 * ks, lane));
                ldsm4t(al, at_addr(sm.A[1], LB64, 16 * w, 16 * ks, lane));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    ldsm4t(b, bk_addr(sdO, LB64, 16 * ks, 16 * np, lane));
                    mma_x2(a1[2 * np], ah, al, b[0], b[1]);
                    mma_x2(a1[2 * np + 1], ah, al, b[2], b[3]);
                }
            }
#pragma unroll 2
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t ah[4], al[4];
                ldsm4(ah, a_addr(sm.K[0], LB, 16 * w, 16 * ks, lane));
                ldsm4(al, a_addr(sm.K[1], LB, 16 * w, 16 * ks, lane));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t bh[4], bl[4];
                    ldsm4t(bh, bk_addr(sm.dS[0], LB64, 16 * ks, 16 * np, lane));
                    ldsm4t(bl, bk_addr(sm.dS[1], LB64, 16 * ks, 16 * np, lane));
                    mma_x3(a2[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                    mma_x3(a2[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int row = 16 * w + g + 8 * hf, col = 8 * nt + 2 * t;
                    const float d0 = fmaf(p.scale, a1[nt][2 * hf], a2[nt][2 * hf]);
                    const float d1 = fmaf(p.scale, a1[nt][2 * hf + 1], a2[nt][2 * hf + 1]);
                    uint32_t hi, lo;
                    split2(-d0, -d1, hi, lo);
                    *reinterpret_cast<uint32_t*>(&sm.X[0][row * LB64 + col]) = hi;
                    *reinterpret_cast<uint32_t*>(&sm.X[1][row * LB64 + col]) = lo;
                    if (bwd)
                        *reinterpret_cast<float2*>(p.dDelta + chd * CH * D + row * D + col0 + col) =
                            make_float2(d0, d1);
                }
        }
        __syncthreads();
        issue_X(ci - 1);
        // ---- D': dS0 = e^gL dS1 + scale Qg^T dO - W^T dDelta ----
        cp_wait<1>();
        __syncthreads();
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float eg = sm.eGL[32 * w + 16 * mt + g + 8 * (e >> 1)];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) dS[mt][nt][e] *= eg;
            }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            float tq[8][4] = {};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t qh[4], ql[4], wh[4], wl[4];
                ldsm4t(qh, at_addr(sm.Q[0], LB, 32 * w + 16 * mt, 16 * ks, lane));
                ldsm4t(ql, at_addr(sm.Q[1], LB, 32 * w + 16 * mt, 16 * ks, lane));
                ldsm4t(wh, at_addr(sm.W[0], LB, 32 * w + 16 * mt, 16 * ks, lane));
                ldsm4t(wl, at_addr(sm.W[1], LB, 32 * w + 16 * mt, 16 * ks, lane));
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4], xh[4], xl[4];
                    ldsm4t(b, bk_addr(sdO, LB64, 16 * ks, 16 * np, lane));
                    ldsm4t(xh, bk_addr(sm.X[0], LB64, 16 * ks, 16 * np, lane));
                    ldsm4t(xl, bk_addr(sm.X[1], LB64, 16 * ks, 16 * np, lane));
                    mma_x2(tq[2 * np], qh, ql, b[0], b[1]);
                    mma_x2(tq[2 * np + 1], qh, ql, b[2], b[3]);
                    mma_x3(dS[mt][2 * np], wh, wl, xh[0], xh[1], xl[0], xl[1]);
                    mma_x3(dS[mt][2 * np + 1], wh, wl, xh[2], xh[3], xl[2], xl[3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dS[mt][nt][e] = fmaf(p.scale, tq[nt][e], dS[mt][nt][e]);
        }
        __syncthreads();
        issue_Y(ci - 1);
        store_dS();
    }
    cp_wait<0>();
    float* out = bwd ? p.dh0 : p.fragB;
    if (out) {
        out += dh;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int key = 32 * w + 16 * mt + g + 8 * hf, val = col0 + 8 * nt + 2 * t;
                    *reinterpret_cast<float2*>(out + size_t(key) * D + val) =
                        make_float2(dS[mt][nt][2 * hf], dS[mt][nt][2 * hf + 1]);
                }
    }
}

// Per-chunk gradient products that need the chunk's states (tensor cores, 8 warps):
//   dR = Minv^T dDelta, P = dR S0^T, dQg = dO S0^T, dAqk = tril(dO Delta^T),
//   dM = -strict_tril(dR Delta^T), dKb = Delta dS1^T, rsum = rowsum(S0 * dS1).
__global__ void __launch_bounds__(NTHR) k_bwd_gemms(Params p) {
    const int ci = blockIdx.x, h = blockIdx.y;
    if (ci >= *p.nchunks) return;
    const int4 info = p.chunk_tab[ci];
    const int t0 = info.y, L = info.z;
    extern __shared__ __align__(16) unsigned char smraw[];
    BwdGemmSmem& sm = *reinterpret_cast<BwdGemmSmem*>(smraw);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const size_t chd = size_t(ci) * p.H + h;
    const float* S0 = p.sS + chd * D * D;
    const float* dS1 = p.dS1 + chd * D * D;
    const float* Dl = p.sDelta + chd * CH * D;
    const int mt = w & 3, nh = w >> 2;

    cp_tile_bf16(sm.M[0], LB64, p.Mh + chd * CH * CH, CH, CH, CH, tid, NTHR);
    cp_tile_bf16(sm.M[1], LB64, p.Ml + chd * CH * CH, CH, CH, CH, tid, NTHR);
    for (int i = tid; i < CH * 16; i += NTHR) {
        const int r = i >> 4, c = (i & 15) * 8;
        const bool ok = r < L;
        const size_t row = size_t(t0 + (ok ? r : 0));
        cp16z(sm.O + r * LB + c, p.dO + (row * p.H + h) * D + c, ok);
    }
    cp_commit();
    split_tile(sm.X[0], sm.X[1], p.dDelta + chd * CH * D, CH, tid, NTHR);
    split_tile(sm.S[0], sm.S[1], S0, D, tid, NTHR);
    split_tile(sm.Dl[0], sm.Dl[1], Dl, CH, tid, NTHR);
    cp_wait<0>();
    __syncthreads();

    // dR = Minv^T dDelta  [64 tok x 128 val]; warp: tokens 16mt.., values 64nh..
    {
        float acc[8][4] = {};
        for (int ks = mt; ks < 4; ++ks) {  // Minv^T is upper triangular
            uint32_t ah[4], al[4];
            ldsm4t(ah, at_addr(sm.M[0], LB64, 16 * mt, 16 * ks, lane));
            ldsm4t(al, at_addr(sm.M[1], LB64, 16 * mt, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4t(bh, bk_addr(sm.X[0], LB, 16 * ks, 64 * nh + 16 * np, lane));
                ldsm4t(bl, bk_addr(sm.X[1], LB, 16 * ks, 64 * nh + 16 * np, lane));
                mma_x3(acc[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                mma_x3(acc[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
            }
        }
        float* dR = p.dR + chd * CH * D;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = 16 * mt + g + 8 * hf, col = 64 * nh + 8 * nt + 2 * t;
                *reinterpret_cast<float2*>(dR + row * D + col) =
                    make_float2(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
                uint32_t hi, lo;
                split2(acc[nt][2 * hf], acc[nt][2 * hf + 1], hi, lo);
                *reinterpret_cast<uint32_t*>(&sm.R[0][row * LB + col]) = hi;
                *reinterpret_cast<uint32_t*>(&sm.R[1][row * LB + col]) = lo;
            }
    }
    __syncthreads();
    // P = dR S0^T and dQg = dO S0^T  [64 tok x 128 key], contraction over values
    {
        float aP[8][4] = {}, aQ[8][4] = {};
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t rh[4], rl[4], o[4];
            ldsm4(rh, a_addr(sm.R[0], LB, 16 * mt, 16 * ks, lane));
            ldsm4(rl, a_addr(sm.R[1], LB, 16 * mt, 16 * ks, lane));
            ldsm4(o, a_addr(sm.O, LB, 16 * mt, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4(bh, bn_addr(sm.S[0], LB, 16 * ks, 64 * nh + 16 * np, lane));
                ldsm4(bl, bn_addr(sm.S[1], LB, 16 * ks, 64 * nh + 16 * np, lane));
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    mma_x3(aP[2 * np + hh], rh, rl, bh[2 * hh], bh[2 * hh + 1], bl[2 * hh], bl[2 * hh + 1]);
                    mma_x2b(aQ[2 * np + hh], o, bh[2 * hh], bh[2 * hh + 1], bl[2 * hh], bl[2 * hh + 1]);
                }
            }
        }
        float* P = p.P + chd * CH * D;
        float* dQg = p.dQg + chd * CH * D;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = 16 * mt + g + 8 * hf, col = 64 * nh + 8 * nt + 2 * t;
                *reinterpret_cast<float2*>(P + row * D + col) = make_float2(aP[nt][2 * hf], aP[nt][2 * hf + 1]);
                *reinterpret_cast<float2*>(dQg + row * D + col) =
                    make_float2(p.scale * aQ[nt][2 * hf], p.scale * aQ[nt][2 * hf + 1]);
            }
    }
    // dAqk = tril(dO Delta^T), dM = -strict_tril(dR Delta^T)  [64 x 64]; warp: rows 16mt, cols 32nh
    {
        float aA[4][4] = {}, aM[4][4] = {};
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t rh[4], rl[4], o[4];
            ldsm4(rh, a_addr(sm.R[0], LB, 16 * mt, 16 * ks, lane));
            ldsm4(rl, a_addr(sm.R[1], LB, 16 * mt, 16 * ks, lane));
            ldsm4(o, a_addr(sm.O, LB, 16 * mt, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4(bh, bn_addr(sm.Dl[0], LB, 16 * ks, 32 * nh + 16 * np, lane));
                ldsm4(bl, bn_addr(sm.Dl[1], LB, 16 * ks, 32 * nh + 16 * np, lane));
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    mma_x2b(aA[2 * np + hh], o, bh[2 * hh], bh[2 * hh + 1], bl[2 * hh], bl[2 * hh + 1]);
                    mma_x3(aM[2 * np + hh], rh, rl, bh[2 * hh], bh[2 * hh + 1], bl[2 * hh], bl[2 * hh + 1]);
                }
            }
        }
        float* dAqk = p.dAqk + chd * CH * CH;
        float* dM = p.dM + chd * CH * CH;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * mt + g + 8 * (e >> 1), s = 32 * nh + 8 * nt + 2 * t + (e & 1);
                dAqk[r * CH + s] = s <= r ? p.scale * aA[nt][e] : 0.f;
                dM[r * CH + s] = s < r ? -aM[nt][e] : 0.f;
            }
    }
    __syncthreads();
    // dKb = Delta dS1^T  [64 tok x 128 key]; rsum from the fp32 states
    split_tile(sm.S[0], sm.S[1], dS1, D, tid, NTHR);
    for (int i = w; i < D; i += NTHR / 32) {
        float a = 0.f;
        for (int j = lane; j < D; j += 32) a = fmaf(S0[i * D + j], dS1[i * D + j], a);
        a = warp_sum(a);
        if (lane == 0) p.rsum[chd * D + i] = a;
    }
    __syncthreads();
    {
        float acc[8][4] = {};
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t ah[4], al[4];
            ldsm4(ah, a_addr(sm.Dl[0], LB, 16 * mt, 16 * ks, lane));
            ldsm4(al, a_addr(sm.Dl[1], LB, 16 * mt, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bh[4], bl[4];
                ldsm4(bh, bn_addr(sm.S[0], LB, 16 * ks, 64 * nh + 16 * np, lane));
                ldsm4(bl, bn_addr(sm.S[1], LB, 16 * ks, 64 * nh + 16 * np, lane));
                mma_x3(acc[2 * np], ah, al, bh[0], bh[1], bl[0], bl[1]);
                mma_x3(acc[2 * np + 1], ah, al, bh[2], bh[3], bl[2], bl[3]);
            }
        }
        float* dKb = p.dKb + chd * CH * D;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = 16 * mt + g + 8 * hf, col = 64 * nh + 8 * nt + 2 * t;
                *reinterpret_cast<float2*>(dKb + row * D + col) = make_float2(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
            }
    }
}

// Intra-chunk gradients of one (chunk, head): dq, dk, dv, dbeta, dg / da and the partial sums
// of dA_log / ddt_bias.  Warp w owns rows w, w+8, ...; lane owns channels lane + 32 m.
__global__ void __launch_bounds__(NTHR) k_bwd_intra(Params p) {
    const int ci = blockIdx.x, h = blockIdx.y;
    if (ci >= *p.nchunks) return;
    const int4 info = p.chunk_tab[ci];
    const int t0 = info.y, L = info.z;
    extern __shared__ float sm[];
    float* sq = sm;
    float* sk = sq + CH * LDP;
    float* sg = sk + CH * LDP;
    float* sdg = sg + CH * LDP;
    float* sdAqk = sdg + CH * LDP;
    float* sdAkk = sdAqk + CH * LDA;
    float* sAkk = sdAkk + CH * LDA;
    float* sbeta = sAkk + CH * LDA;
    float* srq = sbeta + CH;
    float* srk = srq + CH;
    float* red = srk + CH;  // [NTHR]
    const int tid = threadIdx.x, w = tid / 32, lane = tid % 32;
    const size_t chd = size_t(ci) * p.H + h;

    for (int i = tid; i < CH * D; i += NTHR) {
        const int r = i / D, c = i % D;
        float qv = 0.f, kv = 0.f;
        if (r < L) {
            const size_t off = (size_t(t0 + r) * p.H + h) * D + c;
            qv = bf2f(p.q[off]);
            kv = bf2f(p.k[off]);
        }
        sq[r * LDP + c] = qv;
        sk[r * LDP + c] = kv;
    }
    if (tid < CH) sbeta[tid] = tid < L ? bf2f(p.beta[size_t(t0 + tid) * p.H + h]) : 0.f;
    {
        const float* gam = p.gam + chd * CH * D;
        for (int i = tid; i < CH * D; i += NTHR) sg[(i / D) * LDP + i % D] = gam[i];
    }
    __syncthreads();
    for (int r = w; r < CH; r += NTHR / 32) {
        float ra = 1.f, rb = 1.f;
        if (p.l2n) {
            float a = 0.f, b = 0.f;
            for (int c = lane; c < D; c += 32) {
                float x = sq[r * LDP + c], y = sk[r * LDP + c];
                a = fmaf(x, x, a);
                b = fmaf(y, y, b);
            }
            a = warp_sum(a);
            b = warp_sum(b);
            ra = 1.f / sqrtf(a + p.eps);
            rb = 1.f / sqrtf(b + p.eps);
            for (int c = lane; c < D; c += 32) {
                sq[r * LDP + c] *= ra;
                sk[r * LDP + c] *= rb;
            }
        }
        if (lane == 0) {
            srq[r] = ra;
            srk[r] = rb;
        }
    }
    {
        const float* dAqk = p.dAqk + chd * CH * CH;
        const float* dM = p.dM + chd * CH * CH;
        const float* Akk = p.Akk + chd * CH * CH;
        for (int i = tid; i < CH * CH; i += NTHR) {
            const int r = i / CH, s = i % CH;
            sdAqk[r * LDA + s] = dAqk[i];
            sdAkk[r * LDA + s] = sbeta[r] * dM[i];
            sAkk[r * LDA + s] = Akk[i];
        }
    }
    __syncthreads();

    const float* dQgp = p.dQg + chd * CH * D;
    const float* Pp = p.P + chd * CH * D;
    const float* dKbp = p.dKb + chd * CH * D;
    const float* dRp = p.dR + chd * CH * D;
    const float* dMp = p.dM + chd * CH * CH;
    for (int r = w; r < CH; r += NTHR / 32) {
        const float br = sbeta[r];
        float dqh[4], dkh[4], dbp = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int c = lane + 32 * m;
            const float g = sg[r * LDP + c], gl = sg[(CH - 1) * LDP + c];
            const float er = expf(g), eb = expf(gl - g);
            const float qv = sq[r * LDP + c], kv = sk[r * LDP + c];
            const float dQg = dQgp[r * D + c], Pv = Pp[r * D + c], dKb = dKbp[r * D + c];
            const float dKg = -br * Pv;
            float dq = dQg * er;
            float dk = fmaf(dKg, er, dKb * eb);
            float dgam = dQg * qv * er + dKg * kv * er - dKb * kv * eb;
            float aq = 0.f, ak = 0.f, bq = 0.f, bk = 0.f;
            for (int s = 0; s < r; ++s) {
                const float E = expf(g - sg[s * LDP + c]);
                const float ks = sk[s * LDP + c] * E;
                aq = fmaf(sdAqk[r * LDA + s], ks, aq);
                ak = fmaf(sdAkk[r * LDA + s], ks, ak);
            }
            for (int r2 = r + 1; r2 < CH; ++r2) {
                const float E = expf(sg[r2 * LDP + c] - g);
                bq = fmaf(sdAqk[r2 * LDA + r], sq[r2 * LDP + c] * E, bq);
                bk = fmaf(sdAkk[r2 * LDA + r], sk[r2 * LDP + c] * E, bk);
            }
            const float diag = sdAqk[r * LDA + r];
            dq += aq + diag * kv;
            dk += ak + bq + bk + diag * qv;
            dgam += qv * aq + kv * ak - kv * (bq + bk);
            sdg[r * LDP + c] = dgam;
            dqh[m] = dq;
            dkh[m] = dk;
            // dbeta pieces: dR.v - Kg.P
            const float vv = r < L ? bf2f(p.v[(size_t(t0 + r) * p.H + h) * D + c]) : 0.f;
            const float dRv = dRp[r * D + c];
            dbp += dRv * vv - kv * er * Pv;
            if (r < L) store_out(p.dv, (size_t(t0 + r) * p.H + h) * D + c, br * dRv, p.out_fp32);
        }
        for (int s = lane; s < r; s += 32) dbp += sAkk[r * LDA + s] * dMp[r * CH + s];
        dbp = warp_sum(dbp);
        float pq = 0.f, pk = 0.f;
        if (p.l2n) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                pq += sq[r * LDP + lane + 32 * m] * dqh[m];
                pk += sk[r * LDP + lane + 32 * m] * dkh[m];
            }
            pq = warp_sum(pq);
            pk = warp_sum(pk);
        }
        if (r < L) {
            const size_t base = (size_t(t0 + r) * p.H + h) * D;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int c = lane + 32 * m;
                float dq = dqh[m], dk = dkh[m];
                if (p.l2n) {
                    dq = (dq - sq[r * LDP + c] * pq) * srq[r];
                    dk = (dk - sk[r * LDP + c] * pk) * srk[r];
                }
                store_out(p.dq, base + c, dq, p.out_fp32);
                store_out(p.dk, base + c, dk, p.out_fp32);
            }
            if (lane == 0) store_out(p.dbeta, size_t(t0 + r) * p.H + h, dbp, p.out_fp32);
        }
    }
    __syncthreads();
    // chunk-end gate term, then reverse cumsum over the chunk (thread per channel)
    if (tid < D) {
        const int c = tid;
        const float gl = sg[(CH - 1) * LDP + c];
        float dgl = expf(gl) * p.rsum[chd * D + c];
        for (int r = 0; r < CH; ++r)
            dgl = fmaf(dKbp[r * D + c], sk[r * LDP + c] * expf(gl - sg[r * LDP + c]), dgl);
        sdg[(CH - 1) * LDP + c] += dgl;
        float run = 0.f;
        for (int r = CH - 1; r >= 0; --r) {
            run += sdg[r * LDP + c];
            sdg[r * LDP + c] = run;
        }
    }
    __syncthreads();
    if (!p.gate_raw) {
        for (int i = tid; i < CH * D; i += NTHR) {
            const int r = i / D, c = i % D;
            if (r < L) p.dg[(size_t(t0 + r) * p.H + h) * D + c] = sdg[r * LDP + c];
        }
        return;
    }
    // raw gate: da = dg * (-exp(A_log)) * sigmoid(a + dt_bias); partials of dA_log and ddt_bias
    const float eA = expf(p.A_log[h]);
    float pa = 0.f;
    if (tid < D) {
        const int c = tid;
        const float db = p.dt_bias[h * D + c];
        float pd = 0.f;
        for (int r = 0; r < L; ++r) {
            const size_t off = (size_t(t0 + r) * p.H + h) * D + c;
            const float x = p.g[off] + db;
            const float dg = sdg[r * LDP + c];
            const float gv = -eA * softplus_f(x);
            const float da = dg * (-eA) * sigmoid_f(x);
            p.dg[off] = da;
            pd += da;
            pa = fmaf(dg, gv, pa);
        }
        p.pddt[chd * D + c] = pd;
    }
    red[tid] = pa;
    __syncthreads();
    for (int s = NTHR / 2; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    if (tid == 0) p.pdA[chd] = red[0];
}

// Fixed-order sums of the per-chunk partials: dA_log[h], ddt_bias[h, :].
__global__ void k_param_reduce(Params p) {
    const int h = blockIdx.x, c = threadIdx.x;
    const int nc = *p.nchunks;
    float s = 0.f;
    for (int ci = 0; ci < nc; ++ci) s += p.pddt[(size_t(ci) * p.H + h) * D + c];
    p.ddt_bias[h * D + c] = s;
    if (c == 0) {
        float a = 0.f;
        for (int ci = 0; ci < nc; ++ci) a += p.pdA[size_t(ci) * p.H + h];
        p.dA_log[h] = a;
    }
}

}  // namespace kda
