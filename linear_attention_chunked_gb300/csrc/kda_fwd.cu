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

// Intra-chunk products of one (chunk, head): gam, Akk, Aqk, Minv, W, U, Qg, Kb.
// Shared: q, k, gam, scratch [64 x 129] fp32; Akk, Aqk, Minv [64 x 65]; beta; gemm scratch.
__global__ void __launch_bounds__(NTHR) k_intra_fwd(Params p) {
    const int ci = blockIdx.x, h = blockIdx.y;
    if (ci >= *p.nchunks) return;
    const int4 info = p.chunk_tab[ci];
    const int t0 = info.y, L = info.z;
    extern __shared__ float sm[];
    float* sq = sm;
    float* sk = sq + CH * LDP;
    float* sg = sk + CH * LDP;
    float* sb = sg + CH * LDP;
    float* sAkk = sb + CH * LDP;
    float* sAqk = sAkk + CH * LDA;
    float* sMi = sAqk + CH * LDA;
    float* sbeta = sMi + CH * LDA;
    float* gs = sbeta + CH;
    const int tid = threadIdx.x;
    const size_t chd = size_t(ci) * p.H + h;

    // 1. loads (zero-padded past the document end), gate
    for (int i = tid; i < CH * D; i += NTHR) {
        const int r = i / D, c = i % D;
        float qv = 0.f, kv = 0.f, gv = 0.f;
        if (r < L) {
            const size_t off = (size_t(t0 + r) * p.H + h) * D + c;
            qv = bf2f(p.q[off]);
            kv = bf2f(p.k[off]);
            const float x = p.g[off];
            gv = p.gate_raw ? -expf(p.A_log[h]) * softplus_f(x + p.dt_bias[h * D + c]) : x;
        }
        sq[r * LDP + c] = qv;
        sk[r * LDP + c] = kv;
        sg[r * LDP + c] = gv;
    }
    if (tid < CH) sbeta[tid] = tid < L ? bf2f(p.beta[size_t(t0 + tid) * p.H + h]) : 0.f;
    __syncthreads();

    // 2. fused L2 norm of q and k over the 128 channels of the head (warp per row)
    if (p.l2n) {
        const int w = tid / 32, lane = tid % 32;
        for (int r = w; r < CH; r += NTHR / 32) {
            float a = 0.f, b = 0.f;
            for (int c = lane; c < D; c += 32) {
                float x = sq[r * LDP + c], y = sk[r * LDP + c];
                a = fmaf(x, x, a);
                b = fmaf(y, y, b);
            }
            a = warp_sum(a);
            b = warp_sum(b);
            const float ra = 1.f / sqrtf(a + p.eps), rb = 1.f / sqrtf(b + p.eps);
            for (int c = lane; c < D; c += 32) {
                sq[r * LDP + c] *= ra;
                sk[r * LDP + c] *= rb;
            }
        }
    }
    // 3. in-chunk inclusive cumsum of the gate (thread per channel)
    if (tid < D) {
        float run = 0.f;
        for (int r = 0; r < CH; ++r) {
            run += sg[r * LDP + tid];
            sg[r * LDP + tid] = run;
        }
    }
    __syncthreads();

    // 4. Akk (strictly lower) and Aqk (lower incl. diagonal) with exact exponent differences
    for (int i = tid; i < CH * CH; i += NTHR) {
        const int r = i / CH, s = i % CH;
        float akk = 0.f, aqk = 0.f;
        if (s <= r) {
            for (int c = 0; c < D; ++c) {
                const float e = expf(sg[r * LDP + c] - sg[s * LDP + c]);
                const float ks = sk[s * LDP + c] * e;
                akk = fmaf(sk[r * LDP + c], ks, akk);
                aqk = fmaf(sq[r * LDP + c], ks, aqk);
            }
        }
        sAkk[r * LDA + s] = s < r ? akk : 0.f;
        sAqk[r * LDA + s] = aqk;
    }
    __syncthreads();

    // 5. Minv = (I + diag(beta) Akk)^-1 by forward substitution, one column per thread
    if (tid < CH) {
        const int c = tid;
        for (int r = 0; r < CH; ++r) {
            float val = (r == c) ? 1.f : 0.f;
            if (r > c) {
                float acc = 0.f;
                for (int s = c; s < r; ++s) acc = fmaf(sAkk[r * LDA + s], sMi[s * LDA + c], acc);
                val = -sbeta[r] * acc;
            }
            sMi[r * LDA + c] = val;
        }
    }
    // scratch = beta * K * e^gam
    for (int i = tid; i < CH * D; i += NTHR) {
        const int r = i / D, c = i % D;
        sb[r * LDP + c] = sbeta[r] * sk[r * LDP + c] * expf(sg[r * LDP + c]);
    }
    __syncthreads();

    // 6. W = Minv (beta K e^gam), then U = Minv (beta V)
    constexpr int TX = D / 8;  // block_gemm<64,128,4,8> thread map
    const int tx = tid % TX, ty = tid / TX;
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return sMi[m * LDA + kk]; },
                                [&](int kk, int n) { return sb[kk * LDP + n]; }, CH, gs, gs + 16 * CH);
        float* W = p.W + chd * CH * D;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) W[(ty + 16 * i) * D + tx + TX * j] = acc[i][j];
    }
    for (int i = tid; i < CH * D; i += NTHR) {
        const int r = i / D, c = i % D;
        sb[r * LDP + c] = r < L ? sbeta[r] * bf2f(p.v[(size_t(t0 + r) * p.H + h) * D + c]) : 0.f;
    }
    {
        float acc[4][8];
        zero_acc(acc);
        block_gemm<CH, D, 4, 8>(acc, [&](int m, int kk) { return sMi[m * LDA + kk]; },
                                [&](int kk, int n) { return sb[kk * LDP + n]; }, CH, gs, gs + 16 * CH);
        float* U = p.U + chd * CH * D;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) U[(ty + 16 * i) * D + tx + TX * j] = acc[i][j];
    }

    // 7. elementwise products and the small matrices
    {
        float* gam = p.gam + chd * CH * D;
        float* Qg = p.Qg + chd * CH * D;
        float* Kb = p.Kb + chd * CH * D;
        for (int i = tid; i < CH * D; i += NTHR) {
            const int r = i / D, c = i % D;
            const float g = sg[r * LDP + c], gl = sg[(CH - 1) * LDP + c];
            gam[i] = g;
            Qg[i] = sq[r * LDP + c] * expf(g);
            Kb[i] = sk[r * LDP + c] * expf(gl - g);
        }
        float* Aqk = p.Aqk + chd * CH * CH;
        float* Akk = p.Akk + chd * CH * CH;
        float* Mi = p.Minv + chd * CH * CH;
        for (int i = tid; i < CH * CH; i += NTHR) {
            const int r = i / CH, s = i % CH;
            Aqk[i] = sAqk[r * LDA + s];
            Akk[i] = sAkk[r * LDA + s];
            Mi[i] = sMi[r * LDA + s];
        }
    }
}

// Inter-chunk state recurrence of one (document, head, 32-column value slice).
// mode CHAIN_FWD_OUT: S from h0; per chunk save S (and Delta) when p.sS is set, write o; ht.
// mode CHAIN_FRAG_MB: blockIdx.z < NSLICE evolves X = I with zero values (-> M), the rest
//                     evolves Y = 0 with the chunk values (-> B); no output.
__global__ void __launch_bounds__(NTHR) k_chain_fwd(Params p, int mode) {
    constexpr int LS = SLICE + 1;
    const int n = blockIdx.x, h = blockIdx.y, sl = blockIdx.z;
    const bool fragX = (mode == CHAIN_FRAG_MB) && sl < NSLICE;
    const int col0 = (sl % NSLICE) * SLICE;
    extern __shared__ float sm[];
    float* sS = sm;            // [128][33]
    float* sD = sS + D * LS;   // [64][33]
    float* gs = sD + CH * LS;
    const int tid = threadIdx.x;
    const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
    const size_t dh = (size_t(n) * p.H + h) * D * D;

    for (int i = tid; i < D * SLICE; i += NTHR) {
        const int r = i / SLICE, j = i % SLICE;
        float v0 = 0.f;
        if (mode == CHAIN_FRAG_MB) v0 = (fragX && r == col0 + j) ? 1.f : 0.f;
        else if (p.h0) v0 = p.h0[dh + size_t(r) * D + col0 + j];
        sS[r * LS + j] = v0;
    }
    __syncthreads();

    for (int ci = c0; ci < c1; ++ci) {
        const int4 info = p.chunk_tab[ci];
        const int t0 = info.y, L = info.z;
        const size_t chd = size_t(ci) * p.H + h;
        const float* W = p.W + chd * CH * D;
        const float* U = p.U + chd * CH * D;
        const float* Qg = p.Qg + chd * CH * D;
        const float* Kb = p.Kb + chd * CH * D;
        const float* Aqk = p.Aqk + chd * CH * CH;
        const float* gam = p.gam + chd * CH * D;
        if (mode == CHAIN_FWD_OUT && p.sS) {
            float* dst = p.sS + chd * D * D;
            for (int i = tid; i < D * SLICE; i += NTHR) {
                const int r = i / SLICE, j = i % SLICE;
                dst[size_t(r) * D + col0 + j] = sS[r * LS + j];
            }
        }
        // Delta = U - W S   (64 x 32)
        {
            float acc[2][4];
            zero_acc(acc);
            block_gemm<CH, SLICE, 2, 4>(acc, [&](int m, int kk) { return W[m * D + kk]; },
                                        [&](int kk, int nn) { return sS[kk * LS + nn]; }, D, gs,
                                        gs + 16 * CH);
            const int tx = tid % 8, ty = tid / 8;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 32 * i, jj = tx + 8 * j;
                    const float u = fragX ? 0.f : U[r * D + col0 + jj];
                    sD[r * LS + jj] = u - acc[i][j];
                }
        }
        __syncthreads();
        if (mode == CHAIN_FWD_OUT) {
            if (p.sDelta) {
                float* dst = p.sDelta + chd * CH * D;
                for (int i = tid; i < CH * SLICE; i += NTHR) {
                    const int r = i / SLICE, j = i % SLICE;
                    dst[r * D + col0 + j] = sD[r * LS + j];
                }
            }
        }
        if (mode == CHAIN_FWD_OUT && p.o) {
            // O = Qg S + Aqk Delta
            float acc[2][4];
            zero_acc(acc);
            block_gemm<CH, SLICE, 2, 4>(acc, [&](int m, int kk) { return Qg[m * D + kk]; },
                                        [&](int kk, int nn) { return sS[kk * LS + nn]; }, D, gs,
                                        gs + 16 * CH);
            block_gemm<CH, SLICE, 2, 4>(acc, [&](int m, int kk) { return Aqk[m * CH + kk]; },
                                        [&](int kk, int nn) { return sD[kk * LS + nn]; }, CH, gs,
                                        gs + 16 * CH);
            const int tx = tid % 8, ty = tid / 8;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 32 * i, jj = tx + 8 * j;
                    if (r < L)
                        store_out(p.o, (size_t(t0 + r) * p.H + h) * D + col0 + jj,
                                  p.scale * acc[i][j], p.out_fp32);
                }
        }
        // S = e^gL S + Kb^T Delta   (128 x 32)
        {
            float acc[4][4];
            zero_acc(acc);
            block_gemm<D, SLICE, 4, 4>(acc, [&](int m, int kk) { return Kb[kk * D + m]; },
                                       [&](int kk, int nn) { return sD[kk * LS + nn]; }, CH, gs,
                                       gs + 16 * D);
            const int tx = tid % 8, ty = tid / 8;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 32 * i, jj = tx + 8 * j;
                    const float e = expf(gam[(CH - 1) * D + r]);
                    sS[r * LS + jj] = fmaf(e, sS[r * LS + jj], acc[i][j]);
                }
        }
        __syncthreads();
    }
    float* out = nullptr;
    if (mode == CHAIN_FWD_OUT) out = p.ht ? p.ht + dh : nullptr;
    else out = (fragX ? p.fragM : p.fragB) + dh;
    if (out)
        for (int i = tid; i < D * SLICE; i += NTHR) {
            const int r = i / SLICE, j = i % SLICE;
            out[size_t(r) * D + col0 + j] = sS[r * LS + j];
        }
}

}  // namespace kda
