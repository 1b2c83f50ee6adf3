// Internal definitions shared by the CUDA translation units of the KDA library.
//
// Chunked evaluation (chunk C = 64 tokens, restarted at every document start; rows past the end
// of a document are zero-padded: q = k = v = 0, beta = 0, g = 0).  Per chunk and head, with
// gam = in-chunk inclusive cumsum of g and gL = gam[63] (per channel):
//   E[r,s,c] = exp(gam[r,c] - gam[s,c])
//   Akk[r,s] = sum_c k_rc k_sc E[r,s,c] (s < r)        Aqk[r,s] = sum_c q_rc k_sc E[r,s,c] (s <= r)
//   Minv = (I + diag(beta) Akk)^-1,  W = Minv diag(beta) (K * e^gam),  U = Minv diag(beta) V
//   Delta = U - W S,  O = (Q * e^gam) S + Aqk Delta,  S <- e^gL * S + (K * e^(gL - gam))^T Delta
// This is the WY / UT form of the delta rule with per-channel gates (Yang et al. 2024, "Gated
// Delta Networks" and "Gated Linear Attention"), applied here to the KDA recurrence.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"  // include/ is on the include path (build.py)
#include "kda_mma.cuh"

namespace kda {

constexpr int D = 128;       // head dim (keys = values = 128)
constexpr int CH = 64;       // chunk length
constexpr int NTHR = 256;    // threads per block of the chunk kernels
constexpr int SLICE = 32;    // value columns per block of the state-recurrence kernels
constexpr int NSLICE = D / SLICE;
constexpr int LDP = D + 4;   // row stride (floats) of [64 x 128] shared tiles: 16-byte aligned rows,
                             // conflict-free float4 access for row-varying lanes
constexpr int LDA = CH + 1;  // padded row stride of [64 x 64] shared tiles

// Byte offsets of every region of the workspace / saved buffers.  Everything is derived from
// (T, N, H) only, so one allocation serves every pack with the same sizes.
//
// Per (chunk, head) the intra-chunk stage writes the operands of the state recurrence: the MMA
// operands W, Qg = Q e^gam, Kb = K e^(gL - gam), Aqk and Minv as bf16 hi/lo planes (hi + lo carries
// ~16 significant bits), U as fp32 (accumulator initialiser), Akk and gam as fp32, and e^gL.
struct Layout {
    int64_t T;
    int N, H;
    int64_t maxC;  // upper bound of the chunk count: ceil(T/64) + N
    // workspace
    size_t status, nchunks, doc_off, doc_order, chunk_tab;
    size_t dS1, dDelta, dR, P, dQg, dKb, dAqk, dM, rsum;              // backward intermediates
    size_t pdA, pddt;                                                 // parameter partials
    size_t replay;    // replay copy of the saved set
    size_t intra_ws;  // intra products of a forward without saved set / of fragment summaries
    size_t ws_fwd, ws_bwd_saved, ws_bwd_replay, ws_frag;
    // chunk groups (group_chunks = G > 0): at most Gmax groups; per op a region of g_bytes at
    // g_fwd / g_bwd_saved / g_bwd_replay holding the group plan (g_plan: group count, group chunk
    // offsets [Gmax + 1], launch order [Gmax], first group of each document [N + 1]) and the
    // per-group summaries M, B (or C) and start states S_in (or end gradients) [Gmax][H][D][D]
    int G;
    int64_t Gmax;
    size_t g_plan, g_M, g_B, g_S, g_bytes;
    size_t g_fwd, g_bwd_saved, g_bwd_replay;
    // saved set
    size_t sv_S, sv_Delta, sv_gM, saved_bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Offsets inside one "record" of the intra-chunk products (relative to its base).
struct IntraRecord {
    size_t Wh, Wl, Qh, Ql, Kh, Kl, Ah, Al, Mh, Ml, U, Akk, gam, eGL, bytes;
};

inline IntraRecord make_intra_record(size_t CHd) {
    IntraRecord R{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    const size_t tileD = CHd * CH * D, tileC = CHd * CH * CH;
    R.Wh = take(tileD * 2);
    R.Wl = take(tileD * 2);
    R.Qh = take(tileD * 2);
    R.Ql = take(tileD * 2);
    R.Kh = take(tileD * 2);
    R.Kl = take(tileD * 2);
    R.Ah = take(tileC * 2);
    R.Al = take(tileC * 2);
    R.Mh = take(tileC * 2);
    R.Ml = take(tileC * 2);
    R.U = take(tileD * 4);
    R.Akk = take(tileC * 4);
    R.gam = take(tileD * 4);
    R.eGL = take(CHd * D * 4);
    R.bytes = o;
    return R;
}

// The saved forward set = [intra-chunk products | per-chunk start states S_c | write vectors
// Delta_c].  The workspace holds the chunk plan, the backward intermediates, and a private copy of
// the intra products (forward without a saved set, fragment summaries) or of the whole saved set
// (checkpoint replay).
inline Layout make_layout(int64_t T, int N, int H, int G = 0) {
    Layout L{};
    L.T = T;
    L.N = N;
    L.H = H;
    L.maxC = (T + CH - 1) / CH + N;
    L.G = G;
    // a document of c chunks has max(1, ceil(c / G)) groups: at most N + ceil(maxC / G) in all
    L.Gmax = G > 0 ? N + (L.maxC + G - 1) / G : 0;
    const size_t CHd = size_t(L.maxC) * H;  // chunk-head pairs
    const size_t tileD = CHd * CH * D, tileC = CHd * CH * CH;
    const size_t gstate = size_t(L.Gmax) * H * D * D * 4;  // one [Gmax][H][D][D] fp32 array
    const IntraRecord R = make_intra_record(CHd);
    // saved set (+ the groups' transition summaries M for the backward's reverse walk)
    L.sv_S = R.bytes;
    L.sv_Delta = align256(L.sv_S + CHd * D * D * 4);
    L.sv_gM = align256(L.sv_Delta + tileD * 4);
    L.saved_bytes = align256(L.sv_gM + gstate);
    // workspace: header | backward intermediates | replay copy of the saved set.  The forward
    // without a saved set and the fragment summaries keep their intra products right after the
    // header instead (they need no backward intermediates).
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    L.status = take(256);
    L.nchunks = take(sizeof(int));
    L.doc_off = take(sizeof(int) * size_t(N + 1));
    L.doc_order = take(sizeof(int) * size_t(N));
    L.chunk_tab = take(sizeof(int4) * size_t(L.maxC));
    L.intra_ws = o;
    L.ws_fwd = o + R.bytes;
    L.ws_frag = o + R.bytes;
    L.dS1 = take(CHd * D * D * 4);
    L.dDelta = take(tileD * 4);
    L.dR = take(tileD * 4);
    L.P = take(tileD * 4);
    L.dQg = take(tileD * 4);
    L.dKb = take(tileD * 4);
    L.dAqk = take(tileC * 4);
    L.dM = take(tileC * 4);
    L.rsum = take(CHd * 2 * D * 4);  // [chunk-head][2 partials][key]
    L.pdA = take(CHd * 4);
    L.pddt = take(CHd * D * 4);
    L.ws_bwd_saved = o;
    L.replay = take(L.saved_bytes);
    L.ws_bwd_replay = o;
    if (G > 0) {  // group region appended to each op's workspace
        size_t g = 0;
        auto gtake = [&](size_t bytes) { size_t at = g; g = align256(g + bytes); return at; };
        L.g_plan = gtake(sizeof(int) * size_t(1 + (L.Gmax + 1) + L.Gmax + (N + 1)));
        L.g_M = gtake(gstate);
        L.g_B = gtake(gstate);
        L.g_S = gtake(gstate);
        L.g_bytes = g;
        L.g_fwd = align256(L.ws_fwd);
        L.ws_fwd = L.g_fwd + g;
        L.g_bwd_saved = align256(L.ws_bwd_saved);
        L.ws_bwd_saved = L.g_bwd_saved + g;
        L.g_bwd_replay = align256(L.ws_bwd_replay);
        L.ws_bwd_replay = L.g_bwd_replay + g;
    }
    return L;
}

// The group plan of a call with chunk groups (device arrays inside the group region).
struct GroupPlan {
    int* ngroups;     // [1]
    int* gdoc_off;    // [Gmax + 1] first chunk of each group (empty groups after the last)
    int* gdoc_order;  // [Gmax] groups by decreasing chunk count
    int* doc_frag;    // [N + 1] first group of each document
    int G, Gmax;
};

// Everything a kernel needs, passed by value.
struct Params {
    int64_t T;
    int N, H;
    int gate_raw, l2n, out_fp32;
    float scale, eps;
    const int* cu;
    const __nv_bfloat16 *q, *k, *v, *beta, *dO;
    const float *g, *A_log, *dt_bias, *h0, *dht;
    void *o, *dq, *dk, *dv, *dbeta;  // fp32 or bf16 per out_fp32
    float *ht, *dg, *dA_log, *ddt_bias, *dh0;
    // workspace regions
    int* status;
    int* nchunks;
    int* doc_off;
    int* doc_order;   // documents by decreasing chunk count (ties: index order)
    int4* chunk_tab;  // {doc, first token, length, chunk index within the doc}
    __nv_bfloat16 *Wh, *Wl, *Qh, *Ql, *Kh, *Kl, *Ah, *Al, *Mh, *Ml;
    float *U, *Akk, *gam, *eGL;
    // per (chunk, head) chunk-end gradient dS1 [2][128][128] and dDelta [2][64][128]: bf16 hi/lo
    // planes (plane 0 = hi, plane 1 = lo), i.e. the split the per-chunk GEMMs consume
    __nv_bfloat16 *dS1, *dDelta;
    float *dR, *P, *dQg, *dKb, *dAqk, *dM, *rsum, *pdA, *pddt;
    // saved set: chunk-start states S_c [2][128][128] and write vectors Delta_c [2][64][128] as
    // bf16 hi/lo planes
    __nv_bfloat16 *sS, *sDelta;
    // fragment summary outputs
    float *fragM, *fragB;
    // saved transition summaries of the chunk groups [Gmax][H][D][D] (group_chunks > 0)
    float* gM;
    int64_t maxC;
};

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Stores four consecutive output elements (index i, a multiple of 4) in the chosen precision.
__device__ __forceinline__ void store_out4(void* base, size_t i, float4 v, int fp32) {
    if (fp32) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + i) = v;
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        memcpy(&u.x, &a, 4);
        memcpy(&u.y, &b, 4);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + i) = u;
    }
}

// Stores an output element in the caller's chosen precision.
__device__ __forceinline__ void store_out(void* base, size_t i, float v, int fp32) {
    if (fp32) static_cast<float*>(base)[i] = v;
    else static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(u), u = e^-|x| in (0, 1].  log1p(u) is taken as
// 2 atanh(z) with z = u / (2 + u) in (0, 1/3]: 2 (z + z^3/3 + ... + z^13/13) has relative
// truncation error below (1/3)^14 / 15 < 1e-7, i.e. FP32-accurate without the library log1p.
__device__ __forceinline__ float softplus_f(float x) {
    const float u = __expf(-fabsf(x));
    const float z = __fdividef(u, 2.f + u), z2 = z * z;
    float pz = fmaf(z2, 1.f / 13.f, 1.f / 11.f);
    pz = fmaf(z2, pz, 1.f / 9.f);
    pz = fmaf(z2, pz, 1.f / 7.f);
    pz = fmaf(z2, pz, 1.f / 5.f);
    pz = fmaf(z2, pz, 1.f / 3.f);
    pz = fmaf(z2, pz, 1.f);
    return fmaxf(x, 0.f) + 2.f * z * pz;
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide fp32 product acc += sum_k A(m,k) B(k,n) over an M x N tile by 256 threads.
// Thread (tx, ty) owns rows ty + TY*i and columns tx + TX*j.  Operands are read through the
// loader functors la(m,k), lb(k,n) into shared tiles of KT rows.  Starts and ends with a barrier.
template <int M, int N, int RM, int RN, class LA, class LB>
__device__ __forceinline__ void block_gemm(float (&acc)[RM][RN], LA la, LB lb, int K, float* sA,
                                           float* sB) {
    constexpr int TX = N / RN, TY = M / RM, KT = 16;
    static_assert(TX * TY == NTHR, "tile shape must use 256 threads");
    const int tid = threadIdx.x, tx = tid % TX, ty = tid / TX;
    for (int k0 = 0; k0 < K; k0 += KT) {
        __syncthreads();
        for (int i = tid; i < KT * M; i += NTHR) {
            int kk = i / M, m = i % M;
            sA[kk * M + m] = (k0 + kk < K) ? la(m, k0 + kk) : 0.f;
        }
        for (int i = tid; i < KT * N; i += NTHR) {
            int kk = i / N, n = i % N;
            sB[kk * N + n] = (k0 + kk < K) ? lb(k0 + kk, n) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < KT; ++kk) {
            float a[RM], b[RN];
#pragma unroll
            for (int i = 0; i < RM; ++i) a[i] = sA[kk * M + ty + TY * i];
#pragma unroll
            for (int j = 0; j < RN; ++j) b[j] = sB[kk * N + tx + TX * j];
#pragma unroll
            for (int i = 0; i < RM; ++i)
#pragma unroll
                for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    __syncthreads();
}

// ---- batched tile loads (every global load of a thread is issued before its first use) ----

// [64][128] rows t0.. of head h of a [T, H, 128] bf16 tensor -> fp32 shared [64][ld]; rows >= L
// read as zero.  256 threads.
__device__ __forceinline__ void load_rows_bf16(float* s, int ld, const __nv_bfloat16* g, int t0,
                                               int L, int H, int h, int tid) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = tid + NTHR * k, r = i >> 4, c8 = (i & 15) * 8;
        v[k] = r < L ? *reinterpret_cast<const uint4*>(g + (size_t(t0 + r) * H + h) * D + c8)
                     : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = tid + NTHR * k, r = i >> 4, c8 = (i & 15) * 8;
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            s[r * ld + c8 + 2 * j] = f.x;
            s[r * ld + c8 + 2 * j + 1] = f.y;
        }
    }
}

// [64][128] rows t0.. of head h of a [T, H, 128] fp32 tensor -> registers (8 float4 per thread,
// element index i = tid + 256 k -> row i / 32, column 4 (i % 32)); rows >= L read as zero.
__device__ __forceinline__ void load_rows_f32(float4 (&v)[8], const float* g, int t0, int L, int H,
                                              int h, int tid) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = tid + NTHR * k, r = i >> 5, c4 = (i & 31) * 4;
        v[k] = r < L ? *reinterpret_cast<const float4*>(g + (size_t(t0 + r) * H + h) * D + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Dense [ROWS][128] fp32 tile -> registers, same element mapping (ROWS / 8 float4 per thread).
template <int ROWS>
__device__ __forceinline__ void load_tile_f32(float4 (&v)[ROWS / 8], const float* g, int tid) {
#pragma unroll
    for (int k = 0; k < ROWS / 8; ++k) v[k] = reinterpret_cast<const float4*>(g)[tid + NTHR * k];
}

template <int RM, int RN>
__device__ __forceinline__ void zero_acc(float (&acc)[RM][RN]) {
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[i][j] = 0.f;
}

// Scratch for block_gemm: KT x (M + N) floats, M + N <= 256.
constexpr int GEMM_SCRATCH = 16 * 256;

// TMA tensor maps of the state-recurrence operands, built on the host for each call over the
// intra-chunk record: every plane is a run of (chunk, head) tiles, tile index = plane start +
// chunk * H + head.
struct TcMaps {
    CUtensorMap m128;  // W, Qg, Kb hi / lo planes as [tile][64 rows][128 bf16]
    CUtensorMap m64;   // Aqk and Minv hi / lo planes as [tile][64 rows][64 bf16]
    CUtensorMap mdO;   // dO [T][H][128] bf16 as 64 x 64 boxes {values, head, tokens} (backward)
    // backward per-chunk operands, tile = 2 * (chunk * H + head) + plane: dDelta and Delta
    // [tile][64][128] (64 x 64 boxes), S_c and dS1 [tile][128][128] (64 x 128 boxes)
    CUtensorMap mDD, mDl, mS, mdS;
    // whole operand images in one load (dimension order = shared-memory order, innermost first):
    //   mA1  [W; Qg] of one plane: {64 columns, 64 rows, type W / Qg, column block, tile}
    //   mKb  Kb, Qg or W, both planes: {64 columns, 64 rows, column block, plane, tile}
    //   mAq  Aqk or Minv, both planes: {64 columns, 64 rows, plane, tile}
    //   mDD5, mDl5  dDelta / Delta, both planes: {64 values, 64 tokens, value block, plane, chunk}
    //   mS5  saved S, both planes: {64 values, 128 keys, value block, plane, chunk}
    CUtensorMap mA1, mKb, mAq, mDD5, mDl5, mS5;
    // stores of the saved set by the 64-column forward recurrence: S_c and Delta_c, both planes of
    // one 64-value block, {64 values, 128 keys or 64 tokens, plane-chunk = 2 chunk-head + plane}
    CUtensorMap mSst, mDst;
    // the same stores of the backward recurrence's dS1 and dDelta planes (workspace)
    CUtensorMap mdSst, mdDst;
    // stores of the forward intra kernel's fp32 products: U [tile][64][128] and Akk [tile][64][64]
    // as 32 x 64 boxes (128-byte swizzle); its bf16 planes go through m128 / m64
    CUtensorMap mU, mAkk;
    // loads of the forward intra kernel: the gate g [T][H][128] fp32 as boxes of 128 channels x 1
    // head x 64 tokens (no swizzle; tokens at or past T read as zero)
    CUtensorMap mg;
    // backward intra-chunk inputs: q, k [T][H][128] bf16 as 64 x 64 boxes {values, head, tokens};
    // dAqk, dM [chunk * H + head][64][64] fp32 as 32 x 64 boxes (128-byte swizzle)
    CUtensorMap mq, mk, mdA, mdM;
    // gam of the saved record [chunk * H + head][64][128] fp32 as 32 x 64 boxes (128-byte swizzle)
    CUtensorMap mgam;
    int zWh, zWl, zQh, zQl, zKh, zKl, zAh, zAl, zMh, zMl;  // first tile of each plane
};

// ---- kernels (defined in the .cu files) and their dynamic shared memory ----
size_t intra_smem_bytes();
size_t bwd_gemm_tc_smem_bytes();
constexpr int CHAIN_THREADS = 256;  // 8 warps per state-recurrence block
constexpr int BI_THREADS = 512;     // threads of the backward intra-chunk kernel
constexpr int INTRA_THREADS = 512;  // threads of the forward intra-chunk kernel
constexpr int NHALF = 2;            // value halves (64 columns) per head in the recurrences
__global__ void k_plan(Params p);
__global__ void k_group_plan(Params p, GroupPlan gp);
__global__ void k_intra_fwd(Params p, const __grid_constant__ TcMaps tm);
// state recurrences (value-width templates, launched through these; sms = the device's SMs)
cudaError_t chain_tc_setup();
void launch_chain_fwd_tc(const Params& p, int mode, const TcMaps& tm, unsigned pairs, int sms,
                         cudaStream_t st);
void launch_chain_bwd_tc(const Params& p, int mode, const TcMaps& tm, unsigned pairs, int sms,
                         cudaStream_t st);
__global__ void k_bwd_gemms_tc(Params p, const __grid_constant__ TcMaps tm);
cudaError_t bwd_intra_setup();  // shared-memory limits of the backward intra kernel
void launch_bwd_intra(const Params& p, const TcMaps& tm, unsigned grid, cudaStream_t st);
__global__ void k_param_reduce(Params p);
__global__ void k_walk(int N, const int* doc_frag, int F, int H, const float* M, const float* B,
                       const float* S0, int reverse, float* S_in, float* S_final);
// tensor-core transfer walks (kda_walk_precision other than KDA_WALK_FP32)
cudaError_t walk_tc_setup();
void launch_walk_tc(int precision, int N, const int* doc_frag, int F, int H, const float* M,
                    const float* B, const float* S0, int reverse, float* S_in, float* S_final,
                    int* status, cudaStream_t st);

// Launch accounting: every kernel launch of the library sits inside a ProfScope, which counts it
// and, while profiling is enabled (kda_profile_enable), brackets it with CUDA events on its stream.
enum KernelKind {
    KK_PLAN, KK_INTRA_FWD, KK_CHAIN_FWD, KK_CHAIN_BWD, KK_BWD_GEMMS, KK_BWD_INTRA,
    KK_PARAM_REDUCE, KK_WALK, KK_CONV_FWD, KK_CONV_BWD, KK_CONV_REDUCE, KK_COUNT
};
const char* kernel_name(int kind);
class ProfScope {
  public:
    ProfScope(int kind, cudaStream_t st);
    ~ProfScope();
  private:
    int kind_;
    cudaStream_t st_;
    cudaEvent_t a_, b_;
};

// chain modes
constexpr int CHAIN_FWD_OUT = 0;   // forward: o, ht, optional saved set
constexpr int CHAIN_FRAG_MB = 1;   // fragment summary: augmented state [M | B]
constexpr int CHAIN_BWD = 0;       // backward: dS1, dDelta, dh0
constexpr int CHAIN_FRAG_C = 1;    // fragment summary backward: C only

}  // namespace kda
