// Width-4 causal depthwise conv1d + SiLU ahead of KDA's q / k / v, forward and backward, over
// documents packed by cu_seqlens (optionally with three halo rows in front of every document).
//
//   z[t, c] = b[c] + sum_{j=0..3} w[c, j] x[t - 3 + j, c],   y = silu(z) = z sigmoid(z)
//
// A read before a document's first token takes the document's halo row, else zero.  Source: the
// KCP transfer-walk page (flashinfer PR #7176), PR description: the module forward runs the conv
// halo exchange and the conv ahead of the KDA recurrence; the family ships a width-4 causal
// conv1d + SiLU training backend with a halo variant.
//
// Both kernels are bound by HBM traffic (2 bytes of x per channel and token in, as much out),
// so they are plain streaming kernels: a thread owns 4 consecutive channels (an 8-byte bf16 row
// segment; a warp covers 128 channels, 256 contiguous bytes of a row) and a run of TT tokens,
// keeps the three previous rows in registers, and streams its rows through a ring of shared
// memory slots filled by cp.async RING - 1 rows ahead, so that enough bytes are in flight per SM
// without holding them in registers.  The backward recomputes z, takes dz = dy silu'(z) for its tokens and the
// three after them (their dz also reaches its last rows), and writes dx of its own rows only;
// dw and db are summed per block in a fixed order and then over blocks by a second kernel, so
// every result is bitwise reproducible (no atomics).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int CV_TX = 32, CV_TY = 8;  // block: 32 channel groups x 8 token runs
constexpr int CV_TT = 64;             // tokens per run
constexpr int CV_RING = 16;           // ring slots per thread (forward): four groups of four rows
constexpr int CV_GR = 4;              // rows per copy group (forward)
constexpr int CV_RING_B = 8;          // ring slots per thread (backward, x and dy)
constexpr int CV_ROWS = CV_TY * CV_TT;  // tokens per block row

struct ConvArgs {
    int64_t T;
    int N, C, act, out_fp32;
    const int* cu;
    const __nv_bfloat16* x;
    const float* w;
    const float* bias;
    const __nv_bfloat16* halo;
    void* y;            // forward output
    const void* dy;     // backward input (dtype of y)
    void* dx;           // backward outputs (dtype of y)
    void* dhalo;
    float* part;        // [row blocks][5][C]: dw0..dw3, db partials
    float *dw, *db;
};

constexpr int CPT = 4;  // channels per thread (8-byte bf16 / 16-byte fp32 row segments)

// 8- and 16-byte cp.async with zero fill (nothing is read when !valid); the source pointer stays
// inside the tensor either way
__device__ __forceinline__ void cp8z(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(valid ? 8 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp16zm(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void bf4_to_f(const uint2& u, float (&f)[CPT]) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
    const float2 v0 = __bfloat1622float2(b[0]), v1 = __bfloat1622float2(b[1]);
    f[0] = v0.x;
    f[1] = v0.y;
    f[2] = v1.x;
    f[3] = v1.y;
}

__device__ __forceinline__ void load_row(const __nv_bfloat16* base, size_t row, int C, int c0,
                                         float (&f)[CPT]) {
    bf4_to_f(*reinterpret_cast<const uint2*>(base + row * size_t(C) + c0), f);
}

// CPT consecutive values of a row of a [rows][C] tensor, fp32 or bf16 storage
__device__ __forceinline__ void store_row(void* base, size_t row, int C, int c0,
                                          const float (&f)[CPT], int fp32) {
    const size_t i = row * size_t(C) + c0;
    if (fp32) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + i) = make_float4(f[0], f[1], f[2], f[3]);
    } else {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + i) =
            make_uint2(pack2(f[0], f[1]), pack2(f[2], f[3]));
    }
}

// logistic function; the fast reciprocal returns 0 once 1 + e^-z exceeds 2^126 (z < -87), the
// limit the exact value has there
__device__ __forceinline__ float sigm(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// Document of token t: the last n with cu[n] <= t among documents that are not empty before t
// (binary search; indices stay inside [0, N - 1] for any cu_seqlens).
__device__ __forceinline__ int doc_of(const int* cu, int N, int t) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int(cu[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The three rows before token t of document n (start s): x rows inside the document, halo rows
// (or zeros) before it.
__device__ __forceinline__ void window_at(const ConvArgs& a, int n, int s, int t, int c0,
                                          float (&xm)[3][CPT]) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int r = t - 3 + i;  // xm[i] = x[t - 3 + i]
        if (r >= s && r >= 0) {
            load_row(a.x, size_t(r), a.C, c0, xm[i]);
        } else if (a.halo) {
            const int hr = int(r - s + 3);  // halo row 0..2 (rows before the document start)
            if (hr >= 0) load_row(a.halo, size_t(n) * 3 + hr, a.C, c0, xm[i]);
            else {
#pragma unroll
                for (int k = 0; k < CPT; ++k) xm[i][k] = 0.f;
            }
        } else {
#pragma unroll
            for (int k = 0; k < CPT; ++k) xm[i][k] = 0.f;
        }
    }
}

__global__ void __launch_bounds__(CV_TX * CV_TY, 3) k_conv_fwd(ConvArgs a) {
    __shared__ uint2 ring[CV_TY][CV_RING][CV_TX];  // [token run][slot][channel group]: one x row each
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int cg = blockIdx.x * CV_TX + tx, c0 = CPT * cg;
    const int t0 = (int(blockIdx.y) * CV_TY + ty) * CV_TT;
    if (c0 >= a.C || t0 >= a.T) return;  // (no block-wide barrier in this kernel)
    const int t1 = min(t0 + CV_TT, int(a.T));
    const size_t C = size_t(a.C);
    const __nv_bfloat16* xcol = a.x + c0;  // row t at xcol + t C
    // group q = rows t0 + 4 q .. t0 + 4 q + 3 into slots 4 (q mod 4) ..; rows past the run are
    // zero-filled and never read
    auto fill = [&](int q) {
        const int tq = t0 + CV_GR * q;
        const __nv_bfloat16* src = xcol + size_t(tq) * C;
#pragma unroll
        for (int j = 0; j < CV_GR; ++j) {
            const bool ok = tq + j < t1;
            cp8z(&ring[ty][(q & 3) * CV_GR + j][tx], ok ? src + j * C : xcol + size_t(t0) * C, ok);
        }
        cp_commit();
    };
    fill(0);
    fill(1);
    fill(2);
    float w[4][CPT], b[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const float4 wk = *reinterpret_cast<const float4*>(a.w + size_t(c0 + k) * 4);
        w[0][k] = wk.x; w[1][k] = wk.y; w[2][k] = wk.z; w[3][k] = wk.w;
        b[k] = a.bias ? a.bias[c0 + k] : 0.f;
    }
    int n = doc_of(a.cu, a.N, t0);
    int s = a.cu[n], e = a.cu[n + 1];
    float xm[3][CPT];
    window_at(a, n, s, t0, c0, xm);
    for (int q = 0; t0 + CV_GR * q < t1; ++q) {
        cp_wait<2>();  // group q has landed (groups q + 1, q + 2 may be in flight)
        uint2 raw[CV_GR];
#pragma unroll
        for (int j = 0; j < CV_GR; ++j) raw[j] = ring[ty][(q & 3) * CV_GR + j][tx];
        fill(q + 3);  // into the slots of group q - 1, read in the previous iteration
#pragma unroll
        for (int j = 0; j < CV_GR; ++j) {
            const int t = t0 + CV_GR * q + j;
            if (t >= t1) break;
            float xr[CPT];
            bf4_to_f(raw[j], xr);
            if (t >= e) {  // next document (skipping empty ones): its halo rows or zeros
                while (n + 1 < a.N && int(a.cu[n + 1]) <= t) ++n;
                s = a.cu[n];
                e = a.cu[n + 1];
                window_at(a, n, s, t, c0, xm);
            }
            float out[CPT];
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const float z = b[k] + w[0][k] * xm[0][k] + w[1][k] * xm[1][k] +
                                w[2][k] * xm[2][k] + w[3][k] * xr[k];
                out[k] = a.act ? __fdividef(z, 1.f + __expf(-z)) : z;
                xm[0][k] = xm[1][k];
                xm[1][k] = xm[2][k];
                xm[2][k] = xr[k];
            }
            store_row(a.y, size_t(t), a.C, c0, out, a.out_fp32);
        }
    }
    cp_wait<0>();  // no copy into the ring is in flight when the thread leaves
}

// Backward: per thread, tokens t0 .. t1 - 1 own their dx rows and their dw / db terms; dz of the
// three tokens after t1 (same document) completes the last rows.  The owner of a document's
// first token also owns the document's halo gradient.  Every branch below depends only on token
// positions, which all lanes of a warp share (lanes differ in channels), so none diverges.
__global__ void __launch_bounds__(CV_TX * CV_TY, 2) k_conv_bwd(ConvArgs a) {
    // rings of x and dy rows during the token loop; the dw / db reduction scratch afterwards
    __shared__ union {
        struct {
            uint2 x[CV_TY][CV_RING_B][CV_TX];
            uint4 g[CV_TY][CV_RING_B][CV_TX];  // dy: fp32 (16 bytes) or bf16 (the first 8)
        } ring;
        float red[CV_TY][5][CPT][CV_TX + 1];
    } sh;
    auto& red = sh.red;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int cg = blockIdx.x * CV_TX + tx, c0 = CPT * cg;
    const int t0 = (int(blockIdx.y) * CV_TY + ty) * CV_TT;
    const bool active = c0 < a.C && t0 < a.T;
    float pw[4][CPT], pb[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        pb[k] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) pw[j][k] = 0.f;
    }
    if (active) {
        const int C = a.C, fp32 = a.out_fp32, act = a.act;
        const int t1 = min(t0 + CV_TT, int(a.T));
        const int tl = min(t1 + 3, int(a.T));  // last token (exclusive) whose dz is needed
        float w[4][CPT], b[CPT];
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const float4 wk = *reinterpret_cast<const float4*>(a.w + size_t(c0 + k) * 4);
            w[0][k] = wk.x; w[1][k] = wk.y; w[2][k] = wk.z; w[3][k] = wk.w;
            b[k] = a.bias ? a.bias[c0 + k] : 0.f;
        }
        int n = doc_of(a.cu, a.N, t0);
        int s = a.cu[n], e = a.cu[n + 1];
        float xm[3][CPT];
        window_at(a, n, s, t0, c0, xm);
        float acc[4][CPT];  // dx of rows t - 3 .. t (acc[j] = row t - 3 + j), shifted per token
        float dh[3][CPT];   // halo gradient of document n (kept when this thread owns its start)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < CPT; ++k) acc[i][k] = 0.f;
#pragma unroll
        for (int i = 0; i < 3; ++i)
#pragma unroll
            for (int k = 0; k < CPT; ++k) dh[i][k] = 0.f;
        bool own_start = s >= t0 && s < t1;
        auto flush_halo = [&]() {
            if (own_start && a.dhalo)
#pragma unroll
                for (int i = 0; i < 3; ++i) store_row(a.dhalo, size_t(n) * 3 + i, C, c0, dh[i], fp32);
        };
        // rows t - 3 .. t - 3 + cnt - 1 (acc[0 .. cnt-1]) of the current document that this thread
        // owns are complete: store them
        auto emit = [&](int t, int cnt) {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int rc = t - 3 + i;
                if (i < cnt && rc >= t0 && rc < t1 && rc >= s)
                    store_row(a.dx, size_t(rc), C, c0, acc[i], fp32);
            }
        };
        const __nv_bfloat16* xcol = a.x + c0;  // row t at xcol + t C
        // rows t0 .. tl - 1 of x and dy through the ring, RING - 1 rows ahead; rows past tl are
        // zero-filled and never read
        auto fill = [&](int tr) {
            const bool ok = tr < tl;
            const size_t row = size_t(ok ? tr : t0);
            const int slot = (tr - t0) & (CV_RING_B - 1);
            cp8z(&sh.ring.x[ty][slot][tx], xcol + row * C, ok);
            if (fp32) cp16zm(&sh.ring.g[ty][slot][tx], static_cast<const float*>(a.dy) + row * C + c0, ok);
            else cp8z(&sh.ring.g[ty][slot][tx], static_cast<const __nv_bfloat16*>(a.dy) + row * C + c0, ok);
            cp_commit();
        };
#pragma unroll
        for (int i = 0; i < CV_RING_B - 1; ++i) fill(t0 + i);
        int t = t0;  // first token not processed
        for (; t < tl; ++t) {
            cp_wait<CV_RING_B - 2>();  // row t has landed
            const int slot = (t - t0) & (CV_RING_B - 1);
            float xr[CPT], gr[CPT];
            bf4_to_f(sh.ring.x[ty][slot][tx], xr);
            if (fp32) {
                const uint4 u = sh.ring.g[ty][slot][tx];
                gr[0] = __uint_as_float(u.x);
                gr[1] = __uint_as_float(u.y);
                gr[2] = __uint_as_float(u.z);
                gr[3] = __uint_as_float(u.w);
            } else {
                const uint4 u = sh.ring.g[ty][slot][tx];
                bf4_to_f(make_uint2(u.x, u.y), gr);
            }
            fill(t + CV_RING_B - 1);  // into the slot of row t - 1, read in the previous iteration
            if (t >= e) {  // next document: rows of the old one are complete, its halo too
                if (t >= t1) break;  // lookahead stops at the end of the document
                emit(t, 3);
                flush_halo();
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < CPT; ++k) acc[i][k] = 0.f;
                while (n + 1 < a.N && a.cu[n + 1] <= t) ++n;
                s = a.cu[n];
                e = a.cu[n + 1];
                own_start = s >= t0 && s < t1;
#pragma unroll
                for (int i = 0; i < 3; ++i)
#pragma unroll
                    for (int k = 0; k < CPT; ++k) dh[i][k] = 0.f;
                window_at(a, n, s, t, c0, xm);
            }
            float dz[CPT];
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const float z = b[k] + w[0][k] * xm[0][k] + w[1][k] * xm[1][k] +
                                w[2][k] * xm[2][k] + w[3][k] * xr[k];
                if (act) {
                    const float sg = sigm(z);
                    dz[k] = gr[k] * sg * (1.f + z * (1.f - sg));
                } else {
                    dz[k] = gr[k];
                }
            }
            if (t < t1) {  // this thread's dw / db terms
#pragma unroll
                for (int k = 0; k < CPT; ++k) {
                    pw[0][k] = fmaf(dz[k], xm[0][k], pw[0][k]);
                    pw[1][k] = fmaf(dz[k], xm[1][k], pw[1][k]);
                    pw[2][k] = fmaf(dz[k], xm[2][k], pw[2][k]);
                    pw[3][k] = fmaf(dz[k], xr[k], pw[3][k]);
                    pb[k] += dz[k];
                }
            }
            // dz[t] reaches rows t - 3 + j: inside the document into dx, before it (the first
            // three tokens of a document, tt = t - s < 3) into halo row j + tt
            const int tt = t - s;
            if (tt >= 3) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k = 0; k < CPT; ++k) acc[j][k] = fmaf(w[j][k], dz[k], acc[j][k]);
            } else {
#pragma unroll
                for (int k = 0; k < CPT; ++k) {
                    acc[3][k] = fmaf(w[3][k], dz[k], acc[3][k]);
                    if (tt == 0) {
                        dh[0][k] = fmaf(w[0][k], dz[k], dh[0][k]);
                        dh[1][k] = fmaf(w[1][k], dz[k], dh[1][k]);
                        dh[2][k] = fmaf(w[2][k], dz[k], dh[2][k]);
                    } else if (tt == 1) {
                        dh[1][k] = fmaf(w[0][k], dz[k], dh[1][k]);
                        dh[2][k] = fmaf(w[1][k], dz[k], dh[2][k]);
                        acc[2][k] = fmaf(w[2][k], dz[k], acc[2][k]);
                    } else {
                        dh[2][k] = fmaf(w[0][k], dz[k], dh[2][k]);
                        acc[1][k] = fmaf(w[1][k], dz[k], acc[1][k]);
                        acc[2][k] = fmaf(w[2][k], dz[k], acc[2][k]);
                    }
                }
            }
            emit(t, 1);  // row t - 3 is complete
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                acc[0][k] = acc[1][k];
                acc[1][k] = acc[2][k];
                acc[2][k] = acc[3][k];
                acc[3][k] = 0.f;
                xm[0][k] = xm[1][k];
                xm[1][k] = xm[2][k];
                xm[2][k] = xr[k];
            }
        }
        cp_wait<0>();  // no copy into the ring is in flight past the loop
        // rows t - 3 .. t - 1 are still held when the loop stops (end of the lookahead, of the
        // document or of the sequence); they are complete
        emit(t, 3);
        flush_halo();
    }
    // dw / db partials: the 8 token runs of the block summed in order, one row per block row (the
    // scratch overlays the rings: every thread is past its loop and its copies)
    __syncthreads();
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
#pragma unroll
        for (int j = 0; j < 4; ++j) red[ty][j][k][tx] = pw[j][k];
        red[ty][4][k][tx] = pb[k];
    }
    __syncthreads();
    if (c0 < a.C) {
        for (int q = ty; q < 5 * CPT; q += CV_TY) {
            const int j = q / CPT, k = q % CPT;
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < CV_TY; ++r) sum += red[r][j][k][tx];
            a.part[(size_t(blockIdx.y) * 5 + j) * a.C + c0 + k] = sum;
        }
    }
}

// dw, db: partials summed over the block rows in order; empty documents get a zero halo gradient
__global__ void k_conv_reduce(ConvArgs a, int rows) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < 5 * a.C) {
        const int j = i / a.C, c = i % a.C;
        float sum = 0.f;
        for (int r = 0; r < rows; ++r) sum += a.part[(size_t(r) * 5 + j) * a.C + c];
        if (j < 4) a.dw[size_t(c) * 4 + j] = sum;
        else if (a.db) a.db[c] = sum;
    }
    if (a.dhalo) {
        const int G = a.C / CPT;
        for (int q = i; q < a.N * 3 * G; q += gridDim.x * blockDim.x) {
            const int n = q / (3 * G), rem = q % (3 * G);
            if (a.cu[n] < a.cu[n + 1]) continue;  // written by the backward kernel
            const float z[CPT] = {0.f, 0.f, 0.f, 0.f};
            store_row(a.dhalo, size_t(n) * 3 + rem / G, a.C, CPT * (rem % G), z, a.out_fp32);
        }
    }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_conv(const kda_conv_problem* p) {
    // token indices stay 32-bit inside the kernels (a thread's run reads up to 67 tokens past its
    // start)
    if (!p || p->T < 0 || p->T > INT32_MAX - 1024 || p->N < 1 || p->N > (1 << 24) || p->C < 8 ||
        p->C % 8 || p->C > (1 << 24))
        return KDA_ERR_INVALID_ARG;
    if ((p->activation != 0 && p->activation != 1) || (p->out_fp32 != 0 && p->out_fp32 != 1))
        return KDA_ERR_INVALID_ARG;
    if (!p->cu_seqlens || (reinterpret_cast<uintptr_t>(p->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

size_t conv_rows(int64_t T) { return size_t((T + CV_ROWS - 1) / CV_ROWS); }

ConvArgs make_conv(const kda_conv_problem* p, const void* x, const float* w, const float* bias,
                   const void* halo) {
    ConvArgs a{};
    a.T = p->T;
    a.N = p->N;
    a.C = p->C;
    a.act = p->activation;
    a.out_fp32 = p->out_fp32;
    a.cu = p->cu_seqlens;
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.w = w;
    a.bias = bias;
    a.halo = static_cast<const __nv_bfloat16*>(halo);
    return a;
}

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_conv_workspace_size(const kda_conv_problem* p, size_t* ws_bytes) {
    if (kda_status s = check_conv(p)) return s;
    if (ws_bytes) *ws_bytes = align256(conv_rows(p->T) * 5 * size_t(p->C) * sizeof(float));
    return KDA_OK;
}

kda_status kda_conv_fwd(const kda_conv_problem* p, const void* x, const float* w,
                        const float* bias, const void* halo, void* y, kda_stream_t stream) {
    if (kda_status s = check_conv(p)) return s;
    if (p->T > 0 && !(x && al16(x) && y && al16(y))) return KDA_ERR_INVALID_ARG;
    if (!w || !al16(w) || (bias && !al16(bias)) || (halo && !al16(halo))) return KDA_ERR_INVALID_ARG;
    if (p->T == 0) return KDA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ConvArgs a = make_conv(p, x, w, bias, halo);
    a.y = y;
    const dim3 grid(unsigned((p->C / CPT + CV_TX - 1) / CV_TX), unsigned(conv_rows(p->T)));
    {
        ProfScope ps(KK_CONV_FWD, st);
        k_conv_fwd<<<grid, dim3(CV_TX, CV_TY), 0, st>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_conv_bwd(const kda_conv_problem* p, const void* x, const float* w,
                        const float* bias, const void* halo, const void* dy, void* dx, float* dw,
                        float* dbias, void* dhalo, void* ws, size_t ws_bytes, kda_stream_t stream) {
    if (kda_status s = check_conv(p)) return s;
    if (p->T > 0 && !(x && al16(x) && dy && al16(dy) && dx && al16(dx))) return KDA_ERR_INVALID_ARG;
    if (!w || !al16(w) || !dw || !al16(dw) || (bias && !al16(bias)) || (halo && !al16(halo)) ||
        (dbias && !al16(dbias)) || (dhalo && !al16(dhalo)) || !ws || !al16(ws))
        return KDA_ERR_INVALID_ARG;
    if (dhalo && !halo) return KDA_ERR_INVALID_ARG;  // a halo gradient needs the halo
    size_t need = 0;
    kda_conv_workspace_size(p, &need);
    if (ws_bytes < need) return KDA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ConvArgs a = make_conv(p, x, w, bias, halo);
    a.dy = dy;
    a.dx = dx;
    a.dhalo = dhalo;
    a.part = static_cast<float*>(ws);
    a.dw = dw;
    a.db = dbias;
    const unsigned rows = unsigned(conv_rows(p->T));
    if (rows > 0) {
        ProfScope ps(KK_CONV_BWD, st);
        k_conv_bwd<<<dim3(unsigned((p->C / CPT + CV_TX - 1) / CV_TX), rows), dim3(CV_TX, CV_TY), 0, st>>>(a);
    }
    {
        ProfScope ps(KK_CONV_REDUCE, st);
        const int n = 5 * p->C;
        k_conv_reduce<<<unsigned((n + 255) / 256), 256, 0, st>>>(a, int(rows));
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
