// Host side of the C ABI declared in include/kda.h: validation, workspace layout, launches.
// No entry point allocates memory or synchronises the device (kda_read_device_status excepted,
// which exists to synchronise).
#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

using namespace kda;

namespace {

const size_t SMEM_INTRA_FWD = intra_smem_bytes();
const size_t SMEM_BWD_GEMMS_TC = bwd_gemm_tc_smem_bytes();
constexpr size_t SMEM_WALK = (D * (SLICE + 1) + GEMM_SCRATCH) * 4;

std::mutex g_mu;
bool g_ready[128];
int g_sms[128];  // multiprocessor count per device (persistent grids)

// Once per device: check it is an sm_103 part and raise the dynamic shared memory limits.
kda_status setup_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= 128) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ready[dev]) return KDA_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (major != 10 || minor != 3) return KDA_ERR_UNSUPPORTED;
    if (cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        g_sms[dev] < 1)
        return KDA_ERR_CUDA;
    struct { const void* f; size_t smem; } attrs[] = {
        {(const void*)k_intra_fwd, SMEM_INTRA_FWD}, {(const void*)k_bwd_gemms_tc, SMEM_BWD_GEMMS_TC},
        {(const void*)k_walk, SMEM_WALK},
    };
    for (auto& a : attrs)
        if (cudaFuncSetAttribute(a.f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(a.smem)) !=
            cudaSuccess)
            return KDA_ERR_CUDA;
    if (bwd_intra_setup() != cudaSuccess || chain_tc_setup() != cudaSuccess ||
        walk_tc_setup() != cudaSuccess)
        return KDA_ERR_CUDA;
    g_ready[dev] = true;
    return KDA_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

kda_status check_problem(const kda_problem* p) {
    if (!p) return KDA_ERR_INVALID_ARG;
    if (p->d != D) return KDA_ERR_UNSUPPORTED;
    if (p->H < 1 || p->H > 65535 || p->N < 1 || p->N > 65535 || p->T < 0 || p->T > INT32_MAX)
        return KDA_ERR_INVALID_ARG;
    if (int64_t(p->N) * p->H * 2 * NHALF > INT32_MAX) return KDA_ERR_UNSUPPORTED;  // 1-D grids
    if (p->gate != KDA_GATE_G && p->gate != KDA_GATE_RAW) return KDA_ERR_INVALID_ARG;
    if (p->l2norm != 0 && p->l2norm != 1) return KDA_ERR_INVALID_ARG;
    if (p->out_fp32 != 0 && p->out_fp32 != 1) return KDA_ERR_INVALID_ARG;
    if (!p->cu_seqlens || (reinterpret_cast<uintptr_t>(p->cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    if (!(p->l2_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
    if (p->group_chunks < 0 || p->group_chunks > (1 << 20)) return KDA_ERR_INVALID_ARG;
    if (p->group_chunks > 0) {  // the group launches' one-dimensional grids
        const Layout L = make_layout(p->T, p->N, p->H, p->group_chunks);
        if (L.Gmax * p->H * 2 * NHALF > INT32_MAX || L.Gmax > INT32_MAX / 2) return KDA_ERR_UNSUPPORTED;
    }
    return KDA_OK;
}

// Required pointers must be non-null and 16-byte aligned; optional ones only aligned.
bool req(const void* ptr) { return ptr && aligned16(ptr); }
bool opt(const void* ptr) { return !ptr || aligned16(ptr); }

kda_status check_inputs(const kda_problem* p, const void* q, const void* k, const void* v,
                        const void* beta, const float* g, const float* A_log,
                        const float* dt_bias) {
    if (p->T > 0 && !(req(q) && req(k) && req(v) && req(g) && opt(beta) && beta))
        return KDA_ERR_INVALID_ARG;
    if (p->gate == KDA_GATE_RAW && !(req(A_log) && req(dt_bias))) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

Params make_params(const kda_problem* pr, const Layout& L, void* ws) {
    Params p{};
    p.T = pr->T;
    p.N = pr->N;
    p.H = pr->H;
    p.gate_raw = pr->gate == KDA_GATE_RAW;
    p.l2n = pr->l2norm;
    p.out_fp32 = pr->out_fp32;
    p.scale = pr->scale;
    p.eps = pr->l2_eps;
    p.cu = pr->cu_seqlens;
    p.maxC = L.maxC;
    char* w = static_cast<char*>(ws);
    p.status = reinterpret_cast<int*>(w + L.status);
    p.nchunks = reinterpret_cast<int*>(w + L.nchunks);
    p.doc_off = reinterpret_cast<int*>(w + L.doc_off);
    p.doc_order = reinterpret_cast<int*>(w + L.doc_order);
    p.chunk_tab = reinterpret_cast<int4*>(w + L.chunk_tab);
    return p;
}

// Points the intra-chunk products and (optionally) the states at a saved-set image at `base`.
void set_saved(Params& p, const Layout& L, char* base, bool states) {
    const IntraRecord R = make_intra_record(size_t(L.maxC) * L.H);
    auto f = [&](size_t off) { return reinterpret_cast<float*>(base + off); };
    auto b = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(base + off); };
    p.Wh = b(R.Wh);
    p.Wl = b(R.Wl);
    p.Qh = b(R.Qh);
    p.Ql = b(R.Ql);
    p.Kh = b(R.Kh);
    p.Kl = b(R.Kl);
    p.Ah = b(R.Ah);
    p.Al = b(R.Al);
    p.Mh = b(R.Mh);
    p.Ml = b(R.Ml);
    p.U = f(R.U);
    p.Akk = f(R.Akk);
    p.gam = f(R.gam);
    p.eGL = f(R.eGL);
    p.sS = states ? b(L.sv_S) : nullptr;
    p.sDelta = states ? b(L.sv_Delta) : nullptr;
    p.gM = states && L.G > 0 ? f(L.sv_gM) : nullptr;
}

// Chunk groups: the group plan and per-group arrays in the group region at `gbase`, and the
// parameters of a launch over groups (groups take the place of documents: their chunk offsets,
// their launch order, Gmax "documents").
struct Groups {
    GroupPlan gp;
    float *M, *B, *S;  // [Gmax][H][D][D]: summaries M, B or C, start states / end gradients
    Params pg;
};
Groups make_groups(const Params& p, const Layout& L, char* gbase) {
    Groups g{};
    int* plan = reinterpret_cast<int*>(gbase + L.g_plan);
    g.gp.ngroups = plan;
    g.gp.gdoc_off = plan + 1;
    g.gp.gdoc_order = plan + 1 + (L.Gmax + 1);
    g.gp.doc_frag = plan + 1 + (L.Gmax + 1) + L.Gmax;
    g.gp.G = L.G;
    g.gp.Gmax = int(L.Gmax);
    g.M = reinterpret_cast<float*>(gbase + L.g_M);
    g.B = reinterpret_cast<float*>(gbase + L.g_B);
    g.S = reinterpret_cast<float*>(gbase + L.g_S);
    g.pg = p;
    g.pg.N = int(L.Gmax);
    g.pg.doc_off = g.gp.gdoc_off;
    g.pg.doc_order = g.gp.gdoc_order;
    return g;
}

void set_bwd_regions(Params& p, const Layout& L, void* ws) {
    char* w = static_cast<char*>(ws);
    auto f = [&](size_t off) { return reinterpret_cast<float*>(w + off); };
    p.dS1 = reinterpret_cast<__nv_bfloat16*>(w + L.dS1);
    p.dDelta = reinterpret_cast<__nv_bfloat16*>(w + L.dDelta);
    p.dR = f(L.dR);
    p.P = f(L.P);
    p.dQg = f(L.dQg);
    p.dKb = f(L.dKb);
    p.dAqk = f(L.dAqk);
    p.dM = f(L.dM);
    p.rsum = f(L.rsum);
    p.pdA = f(L.pdA);
    p.pddt = f(L.pddt);
}

void set_inputs(Params& p, const void* q, const void* k, const void* v, const void* beta,
                const float* g, const float* A_log, const float* dt_bias) {
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.beta = static_cast<const __nv_bfloat16*>(beta);
    p.g = g;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Tensor maps over the intra-chunk record that p points at (3-D: [tile][64 rows][columns], 128-byte
// swizzle, 64 x 64 boxes).  The W, Qg, Kb planes are consecutive runs of CHd tiles, as are the two
// Aqk planes.
kda_status make_tc_maps(const Params& p, const Layout& L, TcMaps* tm) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return KDA_ERR_CUDA;
    const size_t CHd = size_t(L.maxC) * L.H;
    if (6 * CHd > size_t(INT32_MAX)) return KDA_ERR_UNSUPPORTED;
    const IntraRecord R = make_intra_record(CHd);
    const size_t t128 = size_t(CH) * D * 2, t64 = size_t(CH) * CH * 2;
    if (R.Kl + CHd * t128 - R.Wh != 6 * CHd * t128 || R.Ml + CHd * t64 - R.Ah != 4 * CHd * t64)
        return KDA_ERR_UNSUPPORTED;  // planes not contiguous (layout changed)
    tm->zWh = 0;
    tm->zWl = int((R.Wl - R.Wh) / t128);
    tm->zQh = int((R.Qh - R.Wh) / t128);
    tm->zQl = int((R.Ql - R.Wh) / t128);
    tm->zKh = int((R.Kh - R.Wh) / t128);
    tm->zKl = int((R.Kl - R.Wh) / t128);
    tm->zAh = 0;
    tm->zAl = int((R.Al - R.Ah) / t64);
    tm->zMh = int((R.Mh - R.Ah) / t64);
    tm->zMl = int((R.Ml - R.Ah) / t64);
    const cuuint32_t box[3] = {64, 64, 1}, es[3] = {1, 1, 1};
    const cuuint64_t d128[3] = {D, CH, 6 * CHd}, s128[2] = {D * 2, t128};
    const cuuint64_t d64[3] = {CH, CH, 4 * CHd}, s64[2] = {CH * 2, t64};
    if (enc(&tm->m128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.Wh, d128, s128, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tm->m64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.Ah, d64, s64, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KDA_ERR_CUDA;
    // multi-block images: the extra dimensions step through column blocks (128 B), planes (CHd
    // tiles) and W -> Qg (2 CHd tiles) inside the same record
    const cuuint32_t es5[5] = {1, 1, 1, 1, 1};
    const cuuint32_t b5[5] = {64, 64, 2, 2, 1}, b4[4] = {64, 64, 2, 1};
    const cuuint64_t dA1[5] = {64, CH, 2, 2, 6 * CHd};
    const cuuint64_t sA1[4] = {D * 2, 2 * CHd * t128, 128, t128};
    const cuuint64_t dKb[5] = {64, CH, 2, 2, 6 * CHd};
    const cuuint64_t sKb[4] = {D * 2, 128, CHd * t128, t128};
    const cuuint64_t dAq[4] = {CH, CH, 2, 4 * CHd};
    const cuuint64_t sAq[3] = {CH * 2, CHd * t64, t64};
    if (enc(&tm->mA1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, p.Wh, dA1, sA1, b5, es5,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tm->mKb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, p.Wh, dKb, sKb, b5, es5,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tm->mAq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.Ah, dAq, sAq, b4, es5,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KDA_ERR_CUDA;
    {  // fp32 products of the forward intra kernel (TMA stores)
        const cuuint32_t bF[3] = {32, 64, 1};
        const cuuint64_t dU[3] = {D, CH, CHd}, sU[2] = {D * 4, size_t(CH) * D * 4};
        const cuuint64_t dK[3] = {CH, CH, CHd}, sK[2] = {CH * 4, size_t(CH) * CH * 4};
        if (enc(&tm->mU, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.U, dU, sU, bF, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            enc(&tm->mAkk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.Akk, dK, sK, bF, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    }
    if (L.T > 0) {  // the gate, loaded by the forward intra kernel
        const cuuint32_t bg[3] = {D, 1, CH};
        const cuuint64_t dg[3] = {D, cuuint64_t(L.H), cuuint64_t(L.T)};
        const cuuint64_t sg[2] = {D * 4, cuuint64_t(L.H) * D * 4};
        if (enc(&tm->mg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.g), dg, sg, bg, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    }
    if (p.sS) {  // the saved states and write vectors, stored from the recurrence's shared tiles
        const cuuint32_t bS[3] = {64, 128, 2}, bD[3] = {64, 64, 2};
        const cuuint64_t dS[3] = {D, D, 2 * CHd}, sSt[2] = {D * 2, size_t(D) * D * 2};
        const cuuint64_t dD[3] = {D, CH, 2 * CHd}, sDt[2] = {D * 2, size_t(CH) * D * 2};
        if (enc(&tm->mSst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.sS, dS, sSt, bS, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            enc(&tm->mDst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.sDelta, dD, sDt, bD, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

// Tensor map of dO [T][H][128] bf16: boxes of 64 values x 1 head x 64 tokens (128-byte swizzle);
// tokens at or past T read as zero.
kda_status make_dO_map(const void* dO, int64_t T, int H, TcMaps* tm) {
    if (T <= 0) return KDA_OK;  // no chunks: the map is never used
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return KDA_ERR_CUDA;
    const cuuint32_t box[3] = {64, 1, 64}, es[3] = {1, 1, 1};
    const cuuint64_t dims[3] = {D, cuuint64_t(H), cuuint64_t(T)};
    const cuuint64_t strides[2] = {D * 2, cuuint64_t(H) * D * 2};
    if (enc(&tm->mdO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dO), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

// Tensor maps of the backward per-chunk operands (p's saved set and backward regions set).
kda_status make_bwd_maps(const Params& p, const Layout& L, TcMaps* tm) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return KDA_ERR_CUDA;
    const size_t CHd = size_t(L.maxC) * L.H;
    const cuuint32_t es[3] = {1, 1, 1};
    const cuuint32_t b64[3] = {64, 64, 1}, b128[3] = {64, 128, 1};
    const cuuint64_t d64[3] = {D, CH, 2 * CHd}, s64[2] = {D * 2, size_t(CH) * D * 2};
    const cuuint64_t d128[3] = {D, D, 2 * CHd}, s128[2] = {D * 2, size_t(D) * D * 2};
    struct {
        CUtensorMap* m;
        const void* base;
        const cuuint64_t* dims;
        const cuuint64_t* st;
        const cuuint32_t* box;
    } v[4] = {{&tm->mDD, p.dDelta, d64, s64, b64}, {&tm->mDl, p.sDelta, d64, s64, b64},
              {&tm->mS, p.sS, d128, s128, b128}, {&tm->mdS, p.dS1, d128, s128, b128}};
    for (auto& x : v)
        if (enc(x.m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x.base), x.dims, x.st,
                x.box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    // both planes and both value blocks of one chunk in a single load
    const cuuint32_t es5[5] = {1, 1, 1, 1, 1};
    const cuuint32_t b5d[5] = {64, 64, 2, 2, 1}, b5s[5] = {64, 128, 2, 2, 1};
    const cuuint64_t dd5[5] = {64, CH, 2, 2, CHd}, sd5[4] = {D * 2, 128, size_t(CH) * D * 2, 2 * size_t(CH) * D * 2};
    const cuuint64_t ds5[5] = {64, D, 2, 2, CHd}, ss5[4] = {D * 2, 128, size_t(D) * D * 2, 2 * size_t(D) * D * 2};
    struct {
        CUtensorMap* m;
        const void* base;
        const cuuint64_t* dims;
        const cuuint64_t* st;
        const cuuint32_t* box;
    } v5[3] = {{&tm->mDD5, p.dDelta, dd5, sd5, b5d}, {&tm->mDl5, p.sDelta, dd5, sd5, b5d},
               {&tm->mS5, p.sS, ds5, ss5, b5s}};
    for (auto& x : v5)
        if (enc(x.m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(x.base), x.dims, x.st,
                x.box, es5, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    // stores of dS1 / dDelta by the backward recurrence: one 64-value block, both planes
    const cuuint32_t bS[3] = {64, 128, 2}, bD[3] = {64, 64, 2};
    if (enc(&tm->mdSst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.dS1, d128, s128, bS, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tm->mdDst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.dDelta, d64, s64, bD, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

// Tensor maps of the backward intra-chunk kernel's inputs: q and k (64 x 64 boxes like dO) and
// the dAqk / dM regions (3-D [chunk-head][64][64] fp32, 32 x 64 boxes).
kda_status make_bwd_intra_maps(const Params& p, const Layout& L, int64_t T, TcMaps* tm) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return KDA_ERR_CUDA;
    const size_t CHd = size_t(L.maxC) * L.H;
    const cuuint32_t es[3] = {1, 1, 1};
    const cuuint32_t bq[3] = {64, 1, 64}, ba[3] = {32, 64, 1};
    const cuuint64_t dq[3] = {D, cuuint64_t(L.H), cuuint64_t(T)}, sq[2] = {D * 2, cuuint64_t(L.H) * D * 2};
    const cuuint64_t da[3] = {CH, CH, CHd}, sa[2] = {CH * 4, size_t(CH) * CH * 4};
    const cuuint64_t dg[3] = {D, CH, CHd}, sg[2] = {D * 4, size_t(CH) * D * 4};
    struct {
        CUtensorMap* m;
        CUtensorMapDataType ty;
        const void* base;
        const cuuint64_t* dims;
        const cuuint64_t* st;
        const cuuint32_t* box;
    } v[5] = {{&tm->mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, dq, sq, bq},
              {&tm->mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, dq, sq, bq},
              {&tm->mdA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dAqk, da, sa, ba},
              {&tm->mdM, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dM, da, sa, ba},
              {&tm->mgam, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.gam, dg, sg, ba}};
    for (auto& x : v)
        if (enc(x.m, x.ty, 3, const_cast<void*>(x.base), x.dims, x.st, x.box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    return KDA_OK;
}

// The state recurrences of the forward (o, ht, saved set) and of the backward: one block per
// (document, head, value part), longest documents first.
int device_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    return g_sms[dev];
}
void launch_chain_fwd(const Params& p, const kda_problem* pr, const TcMaps& tm, cudaStream_t st) {
    launch_chain_fwd_tc(p, CHAIN_FWD_OUT, tm, unsigned(pr->N) * unsigned(pr->H), device_sms(), st);
}
void launch_chain_bwd(const Params& p, const kda_problem* pr, const TcMaps& tm, cudaStream_t st) {
    launch_chain_bwd_tc(p, CHAIN_BWD, tm, unsigned(pr->N) * unsigned(pr->H), device_sms(), st);
}

kda_status launched() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Forward state recurrence over chunk groups: the group plan, the groups' summaries (M into
// Mdst, B) in parallel, the transfer walk into every group's start state (and every document's
// final state, ht), then the groups finished as documents from those start states (o and the
// saved states when p asks for them).
void grouped_chain_fwd(const Params& p, const kda_problem* pr, const Layout& L, char* gbase,
                       float* Mdst, const TcMaps& tm, cudaStream_t st) {
    Groups g = make_groups(p, L, gbase);
    const unsigned gpairs = unsigned(L.Gmax) * unsigned(pr->H);
    {
        ProfScope ps(KK_PLAN, st);
        k_group_plan<<<1, NTHR, 0, st>>>(p, g.gp);
    }
    {
        Params sm = g.pg;
        sm.fragM = Mdst;
        sm.fragB = g.B;
        ProfScope ps(KK_CHAIN_FWD, st);
        launch_chain_fwd_tc(sm, CHAIN_FRAG_MB, tm, gpairs, device_sms(), st);
    }
    {
        ProfScope ps(KK_WALK, st);
        launch_walk_tc(KDA_WALK_BF16X3, pr->N, g.gp.doc_frag, int(L.Gmax), pr->H, Mdst, g.B, p.h0,
                       0, g.S, p.ht, p.status, st);
    }
    {
        Params f = g.pg;
        f.h0 = g.S;
        f.ht = nullptr;
        ProfScope ps(KK_CHAIN_FWD, st);
        launch_chain_fwd_tc(f, CHAIN_FWD_OUT, tm, gpairs, device_sms(), st);
    }
}

// Backward state recurrence over chunk groups: the groups' gradient summaries C in parallel, the
// reverse walk (transposed M from the forward) into every group's end gradient (and every
// document's dh0), then the groups finished as documents from those end gradients (the per-chunk
// gradients dS1 and dDelta).
void grouped_chain_bwd(const Params& p, const kda_problem* pr, const Layout& L, char* gbase,
                       const float* Msrc, const TcMaps& tm, cudaStream_t st) {
    Groups g = make_groups(p, L, gbase);
    const unsigned gpairs = unsigned(L.Gmax) * unsigned(pr->H);
    {
        ProfScope ps(KK_PLAN, st);
        k_group_plan<<<1, NTHR, 0, st>>>(p, g.gp);
    }
    {
        Params c = g.pg;
        c.fragB = g.B;
        ProfScope ps(KK_CHAIN_BWD, st);
        launch_chain_bwd_tc(c, CHAIN_FRAG_C, tm, gpairs, device_sms(), st);
    }
    {
        ProfScope ps(KK_WALK, st);
        launch_walk_tc(KDA_WALK_BF16X3, pr->N, g.gp.doc_frag, int(L.Gmax), pr->H, Msrc, g.B, p.dht,
                       1, g.S, p.dh0, p.status, st);
    }
    {
        Params b = g.pg;
        b.dht = g.S;
        b.dh0 = nullptr;
        ProfScope ps(KK_CHAIN_BWD, st);
        launch_chain_bwd_tc(b, CHAIN_BWD, tm, gpairs, device_sms(), st);
    }
}

// plan + intra-chunk products (shared by every op)
kda_status run_prologue(const Params& p, const TcMaps& tm, cudaStream_t st) {
    {
        ProfScope ps(KK_PLAN, st);
        k_plan<<<1, NTHR, 0, st>>>(p);
    }
    if (p.maxC > 0) {
        ProfScope ps(KK_INTRA_FWD, st);
        int dev = 0;
        cudaGetDevice(&dev);
        const long long items = p.maxC * p.H;
        const unsigned grid = unsigned(items < g_sms[dev] ? items : g_sms[dev]);
        k_intra_fwd<<<grid, INTRA_THREADS, SMEM_INTRA_FWD, st>>>(p, tm);
    }
    return launched();
}

// Scratch of the allocation-free forward (kda_fwd_static_ws): one static array per device that
// loads this library.  In host code the symbol is a host-side stand-in, not a device address: the
// device address is looked up with cudaGetSymbolAddress, with the calling device current, on
// every call (a cheap table lookup), so a device reset that reloads the module and moves the
// array never leaves a stale address behind.
__device__ __align__(256) unsigned char g_static_ws[KDA_STATIC_WS_BYTES];

}  // namespace

extern "C" {

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument (null/misaligned pointer, bad size, H < 1)";
        case KDA_ERR_UNSUPPORTED: return "unsupported (head dim must be 128; device must be sm_103)";
        case KDA_ERR_WORKSPACE: return "workspace or saved buffer too small";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        case KDA_ERR_DEVICE_CHECK:
            return "device-side validation failed (malformed cu_seqlens, or a g-form gate above 0)";
        case KDA_ERR_TOO_LARGE:
            return "problem needs more scratch than the allocation-free forward holds (KDA_STATIC_WS_BYTES)";
    }
    return "unknown status";
}

kda_status kda_workspace_size(const kda_problem* p, int op, size_t* ws_bytes, size_t* saved_bytes) {
    if (kda_status s = check_problem(p)) return s;
    const Layout L = make_layout(p->T, p->N, p->H, p->group_chunks);
    size_t ws = 0;
    switch (op) {
        case KDA_OP_FWD: ws = L.ws_fwd; break;
        case KDA_OP_BWD_SAVED: ws = L.ws_bwd_saved; break;
        case KDA_OP_BWD_REPLAY: ws = L.ws_bwd_replay; break;
        case KDA_OP_FRAGMENT: ws = L.ws_frag; break;
        case KDA_OP_WALK: ws = 0; break;
        default: return KDA_ERR_INVALID_ARG;
    }
    if (ws_bytes) *ws_bytes = ws;
    if (saved_bytes) *saved_bytes = L.saved_bytes;
    return KDA_OK;
}

kda_status kda_fwd(const kda_problem* pr, const void* q, const void* k, const void* v,
                   const void* beta, const float* g_or_a, const float* A_log,
                   const float* dt_bias, const float* h0, void* o, float* ht, void* saved,
                   void* ws, size_t ws_bytes, kda_stream_t stream) {
    if (kda_status s = check_problem(pr)) return s;
    if (kda_status s = check_inputs(pr, q, k, v, beta, g_or_a, A_log, dt_bias)) return s;
    if ((pr->T > 0 && !req(o)) || !opt(h0) || !opt(ht) || !opt(saved) || !req(ws))
        return KDA_ERR_INVALID_ARG;
    const Layout L = make_layout(pr->T, pr->N, pr->H, pr->group_chunks);
    if (ws_bytes < L.ws_fwd) return KDA_ERR_WORKSPACE;
    if (kda_status s = setup_device()) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Params p = make_params(pr, L, ws);
    set_inputs(p, q, k, v, beta, g_or_a, A_log, dt_bias);
    p.h0 = h0;
    p.o = o;
    p.ht = ht;
    if (saved) set_saved(p, L, static_cast<char*>(saved), true);
    else set_saved(p, L, static_cast<char*>(ws) + L.intra_ws, false);
    TcMaps tm{};
    if (kda_status s = make_tc_maps(p, L, &tm)) return s;
    if (kda_status s = run_prologue(p, tm, st)) return s;
    if (L.G > 0) {
        char* gbase = static_cast<char*>(ws) + L.g_fwd;
        grouped_chain_fwd(p, pr, L, gbase, saved ? p.gM : reinterpret_cast<float*>(gbase + L.g_M),
                          tm, st);
    } else {
        ProfScope ps(KK_CHAIN_FWD, st);
        launch_chain_fwd(p, pr, tm, st);
    }
    return launched();
}

kda_status kda_fwd_static_ws(const kda_problem* pr, const void* q, const void* k, const void* v,
                             const void* beta, const float* g_or_a, const float* A_log,
                             const float* dt_bias, const float* h0, void* o, float* ht,
                             kda_stream_t stream) {
    if (kda_status s = check_problem(pr)) return s;
    if (pr->group_chunks != 0) return KDA_ERR_UNSUPPORTED;
    const Layout L = make_layout(pr->T, pr->N, pr->H, pr->group_chunks);
    if (L.ws_fwd > KDA_STATIC_WS_BYTES) return KDA_ERR_TOO_LARGE;
    if (kda_status s = setup_device()) return s;  // the calling thread's device, sm_103 only
    void* ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_static_ws) != cudaSuccess || !ws) return KDA_ERR_CUDA;
    return kda_fwd(pr, q, k, v, beta, g_or_a, A_log, dt_bias, h0, o, ht, nullptr, ws,
                   KDA_STATIC_WS_BYTES, stream);
}

kda_status kda_bwd(const kda_problem* pr, const void* q, const void* k, const void* v,
                   const void* beta, const float* g_or_a, const float* A_log,
                   const float* dt_bias, const float* h0, const void* dO, const float* dht,
                   const void* saved, void* dq, void* dk, void* dv, void* dbeta, float* dg_or_da,
                   float* dA_log, float* ddt_bias, float* dh0, void* ws, size_t ws_bytes,
                   kda_stream_t stream) {
    if (kda_status s = check_problem(pr)) return s;
    if (kda_status s = check_inputs(pr, q, k, v, beta, g_or_a, A_log, dt_bias)) return s;
    if (pr->T > 0 && !(req(dO) && req(dq) && req(dk) && req(dv) && req(dbeta) && req(dg_or_da)))
        return KDA_ERR_INVALID_ARG;
    if (pr->gate == KDA_GATE_RAW && !(req(dA_log) && req(ddt_bias))) return KDA_ERR_INVALID_ARG;
    if (!opt(h0) || !opt(dht) || !opt(dh0) || !opt(saved) || !req(ws)) return KDA_ERR_INVALID_ARG;
    const Layout L = make_layout(pr->T, pr->N, pr->H, pr->group_chunks);
    if (ws_bytes < (saved ? L.ws_bwd_saved : L.ws_bwd_replay)) return KDA_ERR_WORKSPACE;
    if (kda_status s = setup_device()) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Params p = make_params(pr, L, ws);
    set_bwd_regions(p, L, ws);
    set_inputs(p, q, k, v, beta, g_or_a, A_log, dt_bias);
    p.h0 = h0;
    p.dht = dht;
    p.dO = static_cast<const __nv_bfloat16*>(dO);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dbeta = dbeta;
    p.dg = dg_or_da;
    p.dA_log = dA_log;
    p.ddt_bias = ddt_bias;
    p.dh0 = dh0;
    char* sv = saved ? static_cast<char*>(const_cast<void*>(saved))
                     : static_cast<char*>(ws) + L.replay;
    set_saved(p, L, sv, true);
    TcMaps tm{};
    if (kda_status s = make_tc_maps(p, L, &tm)) return s;
    if (kda_status s = make_dO_map(dO, pr->T, pr->H, &tm)) return s;
    if (kda_status s = make_bwd_maps(p, L, &tm)) return s;
    if (L.maxC > 0)
        if (kda_status s = make_bwd_intra_maps(p, L, pr->T, &tm)) return s;
    if (saved) {
        // the saved set already holds the intra products and states: only the chunk plan
        ProfScope ps(KK_PLAN, st);
        k_plan<<<1, NTHR, 0, st>>>(p);
    } else {
        // checkpoint replay: recompute the intra products, the states and the write vectors
        if (kda_status s = run_prologue(p, tm, st)) return s;
        Params r = p;
        r.o = nullptr;
        r.ht = nullptr;
        if (L.G > 0) {
            grouped_chain_fwd(r, pr, L, static_cast<char*>(ws) + L.g_bwd_replay, p.gM, tm, st);
        } else {
            ProfScope ps(KK_CHAIN_FWD, st);
            launch_chain_fwd(r, pr, tm, st);
        }
    }
    if (L.G > 0) {
        grouped_chain_bwd(p, pr, L, static_cast<char*>(ws) + (saved ? L.g_bwd_saved : L.g_bwd_replay),
                          p.gM, tm, st);
    } else {
        ProfScope ps(KK_CHAIN_BWD, st);
        launch_chain_bwd(p, pr, tm, st);
    }
    if (L.maxC > 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        const long long items = L.maxC * pr->H;
        const unsigned grid = unsigned(items < g_sms[dev] ? items : g_sms[dev]);  // persistent
        {
            ProfScope ps(KK_BWD_GEMMS, st);
            k_bwd_gemms_tc<<<grid, NTHR, SMEM_BWD_GEMMS_TC, st>>>(p, tm);
        }
        ProfScope ps(KK_BWD_INTRA, st);
        launch_bwd_intra(p, tm, grid, st);
    }
    if (p.gate_raw) {
        ProfScope ps(KK_PARAM_REDUCE, st);
        k_param_reduce<<<pr->H, 4 * D, 0, st>>>(p);
    }
    return launched();
}

kda_status kda_fragment_summary(const kda_problem* pr, int mode, const void* q, const void* k,
                                const void* v, const void* beta, const float* g_or_a,
                                const float* A_log, const float* dt_bias, const void* dO,
                                float* M, float* B_or_C, void* ws, size_t ws_bytes,
                                kda_stream_t stream) {
    if (kda_status s = check_problem(pr)) return s;
    if (pr->group_chunks != 0) return KDA_ERR_UNSUPPORTED;
    if (kda_status s = check_inputs(pr, q, k, v, beta, g_or_a, A_log, dt_bias)) return s;
    if (mode != KDA_FRAG_FWD && mode != KDA_FRAG_BWD) return KDA_ERR_INVALID_ARG;
    if (!req(B_or_C) || !req(ws)) return KDA_ERR_INVALID_ARG;
    if (mode == KDA_FRAG_FWD && !req(M)) return KDA_ERR_INVALID_ARG;
    if (mode == KDA_FRAG_BWD && pr->T > 0 && !req(dO)) return KDA_ERR_INVALID_ARG;
    const Layout L = make_layout(pr->T, pr->N, pr->H, pr->group_chunks);
    if (ws_bytes < L.ws_frag) return KDA_ERR_WORKSPACE;
    if (kda_status s = setup_device()) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Params p = make_params(pr, L, ws);
    set_inputs(p, q, k, v, beta, g_or_a, A_log, dt_bias);
    p.dO = static_cast<const __nv_bfloat16*>(dO);
    p.fragM = M;
    p.fragB = B_or_C;
    set_saved(p, L, static_cast<char*>(ws) + L.intra_ws, false);
    TcMaps tm{};
    if (kda_status s = make_tc_maps(p, L, &tm)) return s;
    if (mode == KDA_FRAG_BWD)
        if (kda_status s = make_dO_map(dO, pr->T, pr->H, &tm)) return s;
    if (kda_status s = run_prologue(p, tm, st)) return s;
    if (mode == KDA_FRAG_FWD) {
        ProfScope ps(KK_CHAIN_FWD, st);
        launch_chain_fwd_tc(p, CHAIN_FRAG_MB, tm, unsigned(pr->N) * unsigned(pr->H), device_sms(), st);
    } else {
        ProfScope ps(KK_CHAIN_BWD, st);
        launch_chain_bwd_tc(p, CHAIN_FRAG_C, tm, unsigned(pr->N) * unsigned(pr->H), device_sms(), st);
    }
    return launched();
}

kda_status kda_transfer_walk(int32_t N, const int32_t* doc_frag, int32_t F, int32_t H,
                             const float* M, const float* B, const float* S0, int reverse,
                             int precision, float* S_in, float* S_final, void* ws,
                             kda_stream_t stream) {
    if (N < 1 || N > 65535 || H < 1 || H > 65535 || F < 0 || !doc_frag ||
        (reinterpret_cast<uintptr_t>(doc_frag) & 3u))
        return KDA_ERR_INVALID_ARG;
    if (reverse != 0 && reverse != 1) return KDA_ERR_INVALID_ARG;
    if (precision < KDA_WALK_FP32 || precision > KDA_WALK_BF16X3_HW) return KDA_ERR_INVALID_ARG;
    if (F > 0 && !(req(M) && req(B) && req(S_in))) return KDA_ERR_INVALID_ARG;
    if (!opt(S0) || !opt(S_final) || !opt(ws)) return KDA_ERR_INVALID_ARG;
    if (kda_status s = setup_device()) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    {
        ProfScope ps(KK_WALK, st);
        if (precision == KDA_WALK_FP32)
            k_walk<<<dim3(N, H, NSLICE), NTHR, SMEM_WALK, st>>>(N, doc_frag, F, H, M, B, S0,
                                                                 reverse, S_in, S_final);
        else
            launch_walk_tc(precision, N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final,
                           static_cast<int*>(ws), st);
    }
    return launched();
}

namespace kda {
// Self-test of the bounded device-side waits: an mbarrier that nothing completes; the wait gives
// up after limit_ns of global time and the kernel reports KDA_ERR_TIMEOUT in the status word, as
// every kernel's timed-out wait does, and returns (no trap, the context stays usable).
__global__ void k_selftest_wait(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_ns)) status[0] = KDA_ERR_TIMEOUT;
}
}  // namespace kda

kda_status kda_selftest_wait_timeout(void* ws, uint32_t limit_us, kda_stream_t stream) {
    if (!req(ws) || limit_us == 0 || limit_us > 1000000u) return KDA_ERR_INVALID_ARG;
    if (kda_status s = setup_device()) return s;
    k_selftest_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(ws),
                                                                        uint64_t(limit_us) * 1000u);
    return launched();
}

kda_status kda_read_device_status(void* ws, int* device_status, kda_stream_t stream) {
    if (!req(ws) || !device_status) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return KDA_ERR_CUDA;
    *device_status = v;
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
