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

__device__ __forceinline__ float load_dO(const Params& p, int t0, int L, int h, int r, int c) {
    return r < L ? p.scale * bf2f(p.dO[(size_t(t0 + r) * p.H + h) * D + c]) : 0.f;
}

// Reverse state recurrence of one (document, head, value slice).
// mode CHAIN_BWD: dS from dht; per chunk writes dS1 (gradient at the chunk end) and dDelta; dh0.
// mode CHAIN_FRAG_C: dS from zero, dO given; writes C (= dS at the fragment start) to fragB.
__global__ void __launch_bounds__(NTHR) k_chain_bwd(Params p, int mode) {
    constexpr int LS = SLICE + 1;
    const int n = blockIdx.x, h = blockIdx.y, sl = blockIdx.z;
    const int col0 = sl * SLICE;
    extern __shared__ float sm[];
    float* sS = sm;            // dS [128][33]
    float* sD = sS + D * LS;   // dDelta [64][33]
    float* gs = sD + CH * LS;
    const int tid = threadIdx.x;
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;
    for (int i = tid; i < D * SLICE; i += NTHR) {
        const int r = i / SLICE, j = i % SLICE;
        sS[r * LS + j] = (mode == CHAIN_BWD && p.dht) ? p.dht[dh + size_t(r) * D + col0 + j] : 0.f;
    }
    __syncthreads();
    for (int ci = c1 - 1; ci >= c0; --ci) {
        const int4 info = p.chunk_tab[ci];
        const int t0 = info.y, L = info.z;
        const size_t chd = size_t(ci) * p.H + h;
        const float* W = p.W + chd * CH * D;
        const float* Qg = p.Qg + chd * CH * D;
        const float* Kb = p.Kb + chd * CH * D;
        const float* Aqk = p.Aqk + chd * CH * CH;
        const float* gam = p.gam + chd * CH * D;
        if (mode == CHAIN_BWD) {
            float* dst = p.dS1 + chd * D * D;
            for (int i = tid; i < D * SLICE; i += NTHR) {
                const int r = i / SLICE, j = i % SLICE;
                dst[size_t(r) * D + col0 + j] = sS[r * LS + j];
            }
        }
        // dDelta = Aqk^T dO + Kb dS1   (64 x 32)
        {
            float acc[2][4];
            zero_acc(acc);
            block_gemm<CH, SLICE, 2, 4>(acc, [&](int m, int kk) { return Aqk[kk * CH + m]; },
                                        [&](int kk, int nn) { return load_dO(p, t0, L, h, kk, col0 + nn); },
                                        CH, gs, gs + 16 * CH);
            block_gemm<CH, SLICE, 2, 4>(acc, [&](int m, int kk) { return Kb[m * D + kk]; },
                                        [&](int kk, int nn) { return sS[kk * LS + nn]; }, D, gs,
                                        gs + 16 * CH);
            const int tx = tid % 8, ty = tid / 8;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) sD[(ty + 32 * i) * LS + tx + 8 * j] = acc[i][j];
        }
        __syncthreads();
        if (mode == CHAIN_BWD) {
            float* dst = p.dDelta + chd * CH * D;
            for (int i = tid; i < CH * SLICE; i += NTHR) {
                const int r = i / SLICE, j = i % SLICE;
                dst[r * D + col0 + j] = sD[r * LS + j];
            }
        }
        // dS0 = e^gL dS1 + Qg^T dO - W^T dDelta   (128 x 32)
        {
            float a1[4][4], a2[4][4];
            zero_acc(a1);
            zero_acc(a2);
            block_gemm<D, SLICE, 4, 4>(a1, [&](int m, int kk) { return Qg[kk * D + m]; },
                                       [&](int kk, int nn) { return load_dO(p, t0, L, h, kk, col0 + nn); },
                                       CH, gs, gs + 16 * D);
            block_gemm<D, SLICE, 4, 4>(a2, [&](int m, int kk) { return W[kk * D + m]; },
                                       [&](int kk, int nn) { return sD[kk * LS + nn]; }, CH, gs,
                                       gs + 16 * D);
            const int tx = tid % 8, ty = tid / 8;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 32 * i, jj = tx + 8 * j;
                    const float e = expf(gam[(CH - 1) * D + r]);
                    sS[r * LS + jj] = fmaf(e, sS[r * LS + jj], a1[i][j] - a2[i][j]);
                }
        }
        __syncthreads();
    }
    float* out = (mode == CHAIN_BWD) ? (p.dh0 ? p.dh0 + dh : nullptr) : p.fragB + dh;
    if (out)
        for (int i = tid; i < D * SLICE; i += NTHR) {
            const int r = i / SLICE, j = i % SLICE;
            out[size_t(r) * D + col0 + j] = sS[r * LS + j];
        }
}

// Per-chunk gradient products that need the chunk's states: dR, P, dQg, dKb, dAqk, dM, rsum.
__global__ void __launch_bounds__(NTHR) k_bwd_gemms(Params p) {
    const int ci = blockIdx.x, h = blockIdx.y;
    if (ci >= *p.nchunks) return;
    const int4 info = p.chunk_tab[ci];
    const int t0 = info.y, L = info.z;
    extern __shared__ float sm[];
    float* gs = sm;
    const int tid = threadIdx.x;
    const size_t chd = size_t(ci) * p.H + h;
    const float* S0 = p.sS + chd * D * D;
    const float* dS1 = p.dS1 + chd * D * D;
    const float* Dl = p.sDelta + chd * CH * D;
    const float* dDl = p.dDelta + chd * CH * D;
    const float* Mi = p.Minv + chd * CH * CH;
    float* dR = p.dR + chd * CH * D;
    constexpr int TX = D / 8;
    const int tx = tid % TX, ty = tid / TX;
    auto store = [&](float* dst, float (&acc)[4][8]) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[(ty + 16 * i) * D + tx + TX * j] = acc[i][j];
    };
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return Mi[kk * CH + m]; },
                                [&](int kk, int nn) { return dDl[kk * D + nn]; }, CH, gs, gs + 16 * CH);
        store(dR, acc);
    }
    __syncthreads();
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return dR[m * D + kk]; },
                                [&](int kk, int nn) { return S0[nn * D + kk]; }, D, gs, gs + 16 * CH);
        store(p.P + chd * CH * D, acc);
    }
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return load_dO(p, t0, L, h, m, kk); },
                                [&](int kk, int nn) { return S0[nn * D + kk]; }, D, gs, gs + 16 * CH);
        store(p.dQg + chd * CH * D, acc);
    }
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return Dl[m * D + kk]; },
                                [&](int kk, int nn) { return dS1[nn * D + kk]; }, D, gs, gs + 16 * CH);
        store(p.dKb + chd * CH * D, acc);
    }
    {
        constexpr int TX2 = CH / 4;
        const int tx2 = tid % TX2, ty2 = tid / TX2;
        float acc[4][4];
        zero_acc(acc);
        block_gemm<CH, CH, 4, 4>(acc, [&](int m, int kk) { return load_dO(p, t0, L, h, m, kk); },
                                 [&](int kk, int nn) { return Dl[nn * D + kk]; }, D, gs, gs + 16 * CH);
        float* dAqk = p.dAqk + chd * CH * CH;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = ty2 + 16 * i, s = tx2 + TX2 * j;
                dAqk[r * CH + s] = s <= r ? acc[i][j] : 0.f;
            }
        zero_acc(acc);
        block_gemm<CH, CH, 4, 4>(acc, [&](int m, int kk) { return dR[m * D + kk]; },
                                 [&](int kk, int nn) { return Dl[nn * D + kk]; }, D, gs, gs + 16 * CH);
        float* dM = p.dM + chd * CH * CH;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = ty2 + 16 * i, s = tx2 + TX2 * j;
                dM[r * CH + s] = s < r ? -acc[i][j] : 0.f;
            }
    }
    {
        const int w = tid / 32, lane = tid % 32;
        for (int i = w; i < D; i += NTHR / 32) {
            float a = 0.f;
            for (int j = lane; j < D; j += 32) a = fmaf(S0[i * D + j], dS1[i * D + j], a);
            a = warp_sum(a);
            if (lane == 0) p.rsum[chd * D + i] = a;
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
