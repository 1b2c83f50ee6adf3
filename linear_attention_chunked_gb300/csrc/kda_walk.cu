// Transfer walk: composes the fragments' affine maps S_out = M S_in + B along each document.
#include "kda_internal.cuh"

namespace kda {

// One block per (document, head, 32-column slice of the state).  FP32 products with FP32
// accumulation (exact to fp32 rounding; the walk is at most a few 128^3 products per document).
// Documents whose fragment range is malformed (decreasing or outside [0, F], F the host-given
// fragment count that sizes M, B and S_in) are skipped.
__global__ void __launch_bounds__(NTHR) k_walk(int N, const int* doc_frag, int F, int H, const float* M,
                                               const float* B, const float* S0, int reverse,
                                               float* S_in, float* S_final) {
    constexpr int LS = SLICE + 1;
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * SLICE;
    extern __shared__ float sm[];
    float* cur = sm;
    float* gs = cur + D * LS;
    const int tid = threadIdx.x;
    const int f0 = doc_frag[n], f1 = doc_frag[n + 1];
    if (f1 < f0 || f0 < 0 || f1 > F) return;
    const size_t dh = (size_t(n) * H + h) * D * D;
    for (int i = tid; i < D * SLICE; i += NTHR) {
        const int r = i / SLICE, j = i % SLICE;
        cur[r * LS + j] = S0 ? S0[dh + size_t(r) * D + col0 + j] : 0.f;
    }
    __syncthreads();
    const int tx = tid % 8, ty = tid / 8;
    for (int s = 0; s < f1 - f0; ++s) {
        const int f = reverse ? f1 - 1 - s : f0 + s;
        const size_t fh = (size_t(f) * H + h) * D * D;
        const float* Mf = M + fh;
        const float* Bf = B + fh;
        for (int i = tid; i < D * SLICE; i += NTHR) {
            const int r = i / SLICE, j = i % SLICE;
            S_in[fh + size_t(r) * D + col0 + j] = cur[r * LS + j];
        }
        float acc[4][4];
        zero_acc(acc);
        if (reverse)
            block_gemm<D, SLICE, 4, 4>(acc, [&](int m, int kk) { return Mf[kk * D + m]; },
                                       [&](int kk, int nn) { return cur[kk * LS + nn]; }, D, gs,
                                       gs + 16 * D);
        else
            block_gemm<D, SLICE, 4, 4>(acc, [&](int m, int kk) { return Mf[m * D + kk]; },
                                       [&](int kk, int nn) { return cur[kk * LS + nn]; }, D, gs,
                                       gs + 16 * D);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = ty + 32 * i, jj = tx + 8 * j;
                cur[r * LS + jj] = acc[i][j] + Bf[size_t(r) * D + col0 + jj];
            }
        __syncthreads();
    }
    if (S_final)
        for (int i = tid; i < D * SLICE; i += NTHR) {
            const int r = i / SLICE, j = i % SLICE;
            S_final[dh + size_t(r) * D + col0 + j] = cur[r * LS + j];
        }
}

}  // namespace kda
