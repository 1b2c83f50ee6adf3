// Transfer walk on tcgen05 tensor cores: S <- M_f S + B_f along the fragments of a document (and
// the transposed reverse walk dS <- M_f^T dS + C_f), with the FP32 operands split into tensor-core
// parts and the products accumulated in FP32 in tensor memory.
//
// The products of the walk are FP32 128 x 128 x 128.  Each FP32 operand x is written as a sum of
// PARTS tensor-core values x = x_0 + x_1 + ... (x_0 the rounding of x to the operand format, x_1
// the rounding of the remainder, and so on); a product keeps the part products x_i y_j with
// i + j < PARTS (the others sit below the FP32 rounding of the result):
//   kind::tf32, PARTS = 1  plain TF32 (11 significant bits per operand)
//   kind::tf32, PARTS = 2  TF32 hi/lo: hi hi + hi lo + lo hi (three products)
//   kind::f16,  PARTS = 3  BF16x3: three bf16 parts per operand, six products (24 bits)
// One block per (document, head, NW value columns): NW = 128 is the full-width walk, NW = 64 the
// half-width walk with two blocks per (document, head).  The state slice lives in registers
// (thread = one key row x NW / 2 values); per fragment the threads write it out (S_in), split it
// into the B operand, split M_f (or M_f^T) into the A operand, thread 0 issues the MMAs, and the
// threads read D back and add B_f.  M of the next fragment is loaded into registers while the
// MMAs run.  Source of the design choice: the KCP transfer-walk page (flashinfer PR #7176), PR
// description (half-width BF16x3 walk with two CTAs per (segment, head); the previous full-width
// TF32 hi/lo walk; FP32 storage of M, B and the states).
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int WALK_THREADS = 256;

// Both operands are K-major, 128-byte swizzled: a K chunk holds E = 128 / element-size K values
// of every row, rows 128 bytes apart, atoms of 8 rows 1024 bytes apart (see kda_tc.cuh).
template <bool TF32, int PARTS, int NW>
struct WalkCfg {
    static constexpr int ES = TF32 ? 4 : 2;                   // operand element bytes
    static constexpr int E = 128 / ES;                        // K values per 128-byte row
    static constexpr int A_CH = 128 * 128;                    // bytes of one A chunk (128 rows)
    static constexpr int B_CH = NW * 128;                     // bytes of one B chunk (NW rows)
    static constexpr int PASS_BYTES_FULL = PARTS * (A_CH + B_CH) * (128 / E);
    static constexpr int NPASS = PASS_BYTES_FULL > 196608 ? 2 : 1;  // K split to fit the tiles
    static constexpr int KP = 128 / NPASS;                    // K values per pass
    static constexpr int KCH = KP / E;                        // K chunks per pass
    static constexpr int A_PART = A_CH * KCH, B_PART = B_CH * KCH;
    static constexpr int OFF_B = PARTS * A_PART;
    static constexpr int OFF_BAR = OFF_B + PARTS * B_PART;
    static constexpr size_t SMEM = size_t(OFF_BAR) + 64 + 1024;  // + alignment slack of the base
    static_assert(KCH >= 1 && KP % E == 0, "pass must hold whole K chunks");
    static_assert(SMEM <= 232448, "walk tiles above the shared-memory limit");
};

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r & 0xFFFFE000u;  // the TF32 value as an FP32 bit pattern
}

// The PARTS operand values of x (as raw bits: TF32 in 32 bits, bf16 in the low 16 bits).
template <bool TF32, int PARTS>
__device__ __forceinline__ void split_parts(float x, uint32_t (&o)[PARTS]) {
    float r = x;
#pragma unroll
    for (int i = 0; i < PARTS; ++i) {
        if (TF32) {
            o[i] = tf32_bits(r);
            r -= __uint_as_float(o[i]);
        } else {
            const __nv_bfloat16 b = __float2bfloat16_rn(r);
            o[i] = uint32_t(__bfloat16_as_ushort(b));
            r -= __bfloat162float(b);
        }
    }
}

// Byte offset of element (row, k) of a K-major 128-byte-swizzled chunked tile whose chunks hold
// `rows` rows (k already relative to the pass).
template <int ES, int E>
__device__ __forceinline__ uint32_t kmajor_off(int row, int k, int chunk_bytes) {
    const int c = k / E, kl = k % E;
    const int byte = kl * ES, j = byte >> 4;
    return uint32_t(c * chunk_bytes + row * 128 + ((j ^ (row & 7)) << 4) + (byte & 15));
}

template <int ES>
__device__ __forceinline__ void st_part(unsigned char* p, uint32_t v) {
    if (ES == 4) *reinterpret_cast<uint32_t*>(p) = v;
    else *reinterpret_cast<uint16_t*>(p) = uint16_t(v);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Instruction descriptor of kind::tf32 (A and B TF32, K-major, FP32 accumulation).
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

}  // namespace

template <bool TF32, int PARTS, int NW>
__global__ void __launch_bounds__(WALK_THREADS, 1)
    k_walk_tc(int N, const int* doc_frag, int F, int H, const float* M, const float* B,
              const float* S0, int reverse, float* S_in, float* S_final, int* status) {
    using C = WalkCfg<TF32, PARTS, NW>;
    constexpr int VPT = NW / 2;  // value columns per thread
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * NW;
    const int f0 = doc_frag[n], f1 = doc_frag[n + 1];
    if (f1 < f0 || f0 < 0 || f1 > F) return;  // malformed fragment range: document skipped
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = tc::align1024(smraw);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);  // 0: MMAs done, 1: spare
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_BAR + 16);
    volatile int* stopf = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 20);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int qd = w & 3, cc = VPT * (w >> 2);
    const int row = 32 * qd + lane;  // key row of this thread (TMEM lane)
    const size_t dh = (size_t(n) * H + h) * D * D;

    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        *stopf = 0;
        tc::fence_mbar_init();
    }
    if (w == 0) tc::tmem_alloc(tslot, NW);
    float S[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) S[j] = 0.f;
    if (S0) {
        const float4* src = reinterpret_cast<const float4*>(S0 + dh + size_t(row) * D + col0 + cc);
#pragma unroll
        for (int j = 0; j < VPT / 4; ++j) {
            const float4 x = src[j];
            S[4 * j] = x.x;
            S[4 * j + 1] = x.y;
            S[4 * j + 2] = x.z;
            S[4 * j + 3] = x.w;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tslot;
    const uint32_t tD = taddr + (uint32_t(32 * qd) << 16);
    const uint32_t idesc = TF32 ? idesc_tf32(128, NW) : tc::idesc_bf16(128, NW, false, false);
    const uint32_t sA = smem_u32(sm), sB = smem_u32(sm + C::OFF_B);

    // M_f (forward) or M_f^T (reverse) as the A operand: thread t loads 16 float4 of M_f, element
    // index e = t + 256 i -> source row e / 32, columns 4 (e % 32) .. +3 (coalesced rows)
    float4 mreg[16];
    auto load_M = [&](int f) {
        const float4* src = reinterpret_cast<const float4*>(M + (size_t(f) * H + h) * D * D);
#pragma unroll
        for (int i = 0; i < 16; ++i) mreg[i] = src[tid + WALK_THREADS * i];
    };
    const int nsteps = f1 - f0;
    if (nsteps > 0) load_M(reverse ? f1 - 1 : f0);
    uint32_t ph = 0;
    bool aborted = false;

    for (int s = 0; s < nsteps; ++s) {
        const int f = reverse ? f1 - 1 - s : f0 + s;
        const size_t fh = (size_t(f) * H + h) * D * D;
        {  // the state entering this fragment
            float4* dst = reinterpret_cast<float4*>(S_in + fh + size_t(row) * D + col0 + cc);
#pragma unroll
            for (int j = 0; j < VPT / 4; ++j)
                dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        }
        for (int pass = 0; pass < C::NPASS; ++pass) {
            const int kb = pass * C::KP;
            // B operand (K-major: tile row = value column, K = key): this thread's key is K index
            if (row >= kb && row < kb + C::KP) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    uint32_t parts[PARTS];
                    split_parts<TF32, PARTS>(S[j], parts);
                    const uint32_t off = kmajor_off<C::ES, C::E>(cc + j, row - kb, C::B_CH);
#pragma unroll
                    for (int pt = 0; pt < PARTS; ++pt)
                        st_part<C::ES>(sm + C::OFF_B + pt * C::B_PART + off, parts[pt]);
                }
            }
            // A operand: forward A[m][k] = M_f[m][k]; reverse A[m][k] = M_f[k][m]
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = tid + WALK_THREADS * i, sr = e >> 5, sc = 4 * (e & 31);
                const float v4[4] = {mreg[i].x, mreg[i].y, mreg[i].z, mreg[i].w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int m = reverse ? sc + u : sr, k = reverse ? sr : sc + u;
                    if (k < kb || k >= kb + C::KP) continue;
                    uint32_t parts[PARTS];
                    split_parts<TF32, PARTS>(v4[u], parts);
                    const uint32_t off = kmajor_off<C::ES, C::E>(m, k - kb, C::A_CH);
#pragma unroll
                    for (int pt = 0; pt < PARTS; ++pt) st_part<C::ES>(sm + pt * C::A_PART + off, parts[pt]);
                }
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (*stopf) {
                aborted = true;
                break;
            }
            if (tid == 0) {
                // part products x_i y_j with i + j < PARTS, smallest terms first
                uint32_t acc = pass > 0 ? 1u : 0u;
#pragma unroll
                for (int ord = PARTS - 1; ord >= 0; --ord)
#pragma unroll
                    for (int pi = 0; pi <= ord; ++pi) {
                        const int pj = ord - pi;
#pragma unroll
                        for (int c = 0; c < C::KCH; ++c)
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks) {
                                const uint64_t ad = tc::sdesc(sA + pi * C::A_PART + c * C::A_CH + 32 * ks, 16, 1024);
                                const uint64_t bd = tc::sdesc(sB + pj * C::B_PART + c * C::B_CH + 32 * ks, 16, 1024);
                                if (TF32) mma_tf32(taddr, ad, bd, idesc, acc);
                                else tc::mma(taddr, ad, bd, idesc, acc);
                                acc = 1u;
                            }
                    }
                tc::mma_commit(&bar[0]);
            }
            __syncwarp();
            if (pass + 1 == C::NPASS && s + 1 < nsteps) load_M(reverse ? f - 1 : f + 1);
            const bool ok = tc::mbar_wait(&bar[0], ph);
            ph ^= 1u;
            if (!ok) *stopf = 1;
            tc::fence_after_sync();
            __syncthreads();  // every thread saw the MMAs complete before the tiles are rewritten
            if (*stopf) {
                aborted = true;
                break;
            }
        }
        if (aborted) break;
        {  // S = D + B_f
            const float4* bsrc = reinterpret_cast<const float4*>(B + fh + size_t(row) * D + col0 + cc);
#pragma unroll
            for (int j0 = 0; j0 < VPT; j0 += 32) {
                float v[32];
                tc::tmem_ld32(tD + cc + j0, v);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 b4 = bsrc[j0 / 4 + j];
                    S[j0 + 4 * j] = v[4 * j] + b4.x;
                    S[j0 + 4 * j + 1] = v[4 * j + 1] + b4.y;
                    S[j0 + 4 * j + 2] = v[4 * j + 2] + b4.z;
                    S[j0 + 4 * j + 3] = v[4 * j + 3] + b4.w;
                }
            }
            tc::fence_before_sync();
        }
    }
    if (aborted) {
        if (tid == 0) {
            tc::drain_mmas(&bar[1], 100000000ull);
            if (status) status[0] = KDA_ERR_TIMEOUT;
        }
    } else if (S_final) {
        float4* dst = reinterpret_cast<float4*>(S_final + dh + size_t(row) * D + col0 + cc);
#pragma unroll
        for (int j = 0; j < VPT / 4; ++j)
            dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(taddr, NW);
}

namespace {

template <bool TF32, int PARTS, int NW>
cudaError_t walk_attr() {
    return cudaFuncSetAttribute(k_walk_tc<TF32, PARTS, NW>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(WalkCfg<TF32, PARTS, NW>::SMEM));
}

template <bool TF32, int PARTS, int NW>
void walk_launch(int N, const int* doc_frag, int F, int H, const float* M, const float* B,
                 const float* S0, int reverse, float* S_in, float* S_final, int* status,
                 cudaStream_t st) {
    k_walk_tc<TF32, PARTS, NW><<<dim3(N, H, D / NW), WALK_THREADS, WalkCfg<TF32, PARTS, NW>::SMEM,
                                 st>>>(N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final, status);
}

}  // namespace

cudaError_t walk_tc_setup() {
    cudaError_t e = walk_attr<true, 1, 128>();
    if (e == cudaSuccess) e = walk_attr<true, 2, 128>();
    if (e == cudaSuccess) e = walk_attr<false, 3, 128>();
    if (e == cudaSuccess) e = walk_attr<false, 3, 64>();
    return e;
}

void launch_walk_tc(int precision, int N, const int* doc_frag, int F, int H, const float* M,
                    const float* B, const float* S0, int reverse, float* S_in, float* S_final,
                    int* status, cudaStream_t st) {
    switch (precision) {
        case KDA_WALK_TF32:
            walk_launch<true, 1, 128>(N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final, status, st);
            break;
        case KDA_WALK_TF32_HILO:
            walk_launch<true, 2, 128>(N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final, status, st);
            break;
        case KDA_WALK_BF16X3:
            walk_launch<false, 3, 128>(N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final, status, st);
            break;
        default:  // KDA_WALK_BF16X3_HW
            walk_launch<false, 3, 64>(N, doc_frag, F, H, M, B, S0, reverse, S_in, S_final, status, st);
            break;
    }
}

}  // namespace kda
